"""The host-side bank model, pinned to the facts the pages print, then applied
to every shared-memory access of the kernels (no GPU)."""
import os

import pytest

import bank_model as BM

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "banks_pages.txt")


def golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if line:
            name, value, _src = line.split()
            vals[name] = int(value)
    return vals


G = golden()


def test_pages_padded_tile_facts():
    for c in range(32):
        assert BM.conflict_degree(BM.pad_tile_column_read(0, c)) == G["pad0_column_read_degree"]
        assert BM.conflict_degree(BM.pad_tile_column_read(1, c)) == G["pad1_column_read_degree"]
        # width 33: lane t lands in bank (t + c) mod 32
        banks = [(a // 4) % 32 for a in BM.pad_tile_column_read(1, c)]
        assert banks == [(t + c) % 32 for t in range(32)]
    assert 32 * 32 * 4 == G["pad0_tile_bytes"] and 32 * 33 * 4 == G["pad1_tile_bytes"]
    assert (33 % 32) == G["cheatsheet_word33_bank"] == (1 % 32)


def test_pages_sgemm_store_facts():
    deg = lambda bk, stride: max(BM.conflict_degree(BM.sgemm_as_store(bk, stride, j))
                                 for j in range(4))
    assert deg(16, 128) == G["sgemm_bk16_stride128_degree"]
    assert deg(8, 128) == G["sgemm_bk8_stride128_degree"]
    assert deg(16, BM.a_stride(128, 16)) == G["sgemm_bk16_stride130_degree"]
    assert BM.a_stride(128, 16) - 128 == G["a_stride_pad_bk16"]
    assert BM.a_stride(128, 32) - 128 == G["a_stride_pad_bk32"]
    assert BM.a_stride(128, 8) - 128 == G["a_stride_pad_bk8"]
    assert 16 * 128 * 4 == G["as_bytes_bm128_bk16"]
    assert 16 * BM.a_stride(128, 16) * 4 == G["as_bytes_padded_bk16"]
    # the column term (innerColA*4 + j)*130 mod 32 takes {2j, 8+2j, 16+2j, 24+2j}
    for j in range(4):
        assert {((c * 4 + j) * 130) % 32 for c in range(4)} == {2 * j, 8 + 2 * j, 16 + 2 * j,
                                                                24 + 2 * j}


def test_broadcast_is_not_a_conflict():
    assert BM.conflict_degree([0] * 32) == 1
    assert BM.conflict_degree([0, 128] * 16) == 2


def test_padded_tile_predictions_for_other_pads():
    # pad 2: bank (2t + c) mod 32 -> two lanes per bank
    assert max(BM.conflict_degree(BM.pad_tile_column_read(2, c)) for c in range(32)) == 2
    # 16-bit elements: two lanes share a word; pad 2 (one word) is conflict-free
    assert max(BM.conflict_degree(BM.pad_tile_column_read(2, c, esize=2)) for c in range(32)) == 1
    assert max(BM.conflict_degree(BM.pad_tile_column_read(0, c, esize=2)) for c in range(32)) == 16
    for pad in (0, 1, 2):
        assert BM.conflict_degree(BM.pad_tile_row_write(pad)) == 1


@pytest.mark.parametrize("V,MR,MC", [(4, 16, 16), (4, 32, 16), (4, 16, 32), (4, 32, 32),
                                     (8, 16, 16), (8, 32, 16), (8, 16, 32)])
def test_vector_tile_is_conflict_free(V, MR, MC):
    for warp in range(8):
        for k in range(V * MR * MC // 256):
            a = BM.vec_tile_load_store(warp, k, V=V, MC=MC)
            assert BM.conflict_degree(a, 16) == 1
        for j in range(MR * MC // 256):
            for m in range(V):
                assert BM.conflict_degree(BM.vec_tile_read(warp, m, V, MR, MC, j), 16) == 1


@pytest.mark.parametrize("V,MR,MC", [(4, 16, 16), (4, 32, 16), (4, 16, 32), (4, 32, 32),
                                     (8, 16, 16), (8, 32, 16), (8, 16, 32)])
def test_misaligned_input_staging_is_conflict_free(V, MR, MC):
    for warp in range(8):
        for k in range(V * MR * MC // 256):
            assert BM.conflict_degree(BM.vec_tile_staging(warp, k, MC), 16) == 1
            assert BM.conflict_degree(BM.vec_tile_staging(warp, k, MC, next_chunk=True), 16) == 1
        a = BM.vec_tile_staging_helper(warp, V * MR, MC)
        if any(x is not None for x in a):
            assert BM.conflict_degree(a, 16) == 1


def test_vector_tile_without_swizzle_would_conflict():
    # the same micro-block read on a plain row-major tile: 8 lanes, one chunk column
    plain = [((4 * lane + 0) * 16 + 0) * 16 for lane in range(32)]
    assert BM.conflict_degree(plain, 16) == 8


@pytest.mark.parametrize("V", [4, 8])
def test_tma_turnaround_is_conflict_free_in_the_model(V):
    for warp in range(8):
        for m in range(V):
            assert BM.conflict_degree(BM.tma_read(warp, m, V), 16) == 1
            assert BM.conflict_degree(BM.tma_write(warp, m, V), 16) == 1


def test_tma_addresses_cover_each_box_chunk_once():
    for V in (4, 8):
        reads = sorted(a for w in range(8) for m in range(V) for a in BM.tma_read(w, m, V))
        writes = sorted(a for w in range(8) for m in range(V) for a in BM.tma_write(w, m, V))
        expect = list(range(0, 2 * 16 * V * 128, 16))
        assert reads == expect and writes == expect


@pytest.mark.parametrize("V", [4, 8])
def test_rotated_reads_of_the_register_store_pipelines_are_conflict_free(V):
    """The warp-specialised and load-only TMA pipelines read rows in a per-lane
    rotated order so the 8 lanes of each 16-byte phase hit 8 swizzle positions;
    without the rotation the same reads would conflict."""
    ws = [a for w in range(8) for m in range(V) for a in BM.ws_consumer_read(w, m, V)]
    assert sorted(ws) == list(range(0, 2 * 16 * V * 128, 16))   # each slot chunk once
    for w in range(8):
        for m in range(V):
            assert BM.conflict_degree(BM.ws_consumer_read(w, m, V), 16) == 1
    ld = [a for m in range(V) for p in range(2) for a in BM.ldst_read(m, p, V)]
    assert sorted(ld) == list(range(0, 8 * V * 128, 16))          # each box chunk once
    for m in range(V):
        for p in range(2):
            assert BM.conflict_degree(BM.ldst_read(m, p, V), 16) == 1
    # the unrotated order: lanes A = 0..7 of a phase read row V*A + m
    plain = [(V * (lane & 7) + 0) * 128 + (((lane >> 3) ^ ((V * (lane & 7)) & 7)) << 4)
             for lane in range(32)]
    assert BM.conflict_degree(plain, 16) > 1


@pytest.mark.parametrize("MR,NT", [(16, 256), (8, 128)])
def test_bf16_column_gather_banks_range_and_coverage(MR, NT):
    """The bf16 shifted stores gather each aligned output chunk from the shared
    tile one element per input row.  With 8 chunks of an output row per warp
    instruction (64-row tiles) the 32 element reads fall on 32 distinct banks;
    with 16 (128-row tiles, 256-byte store runs) two lanes share each bank.
    That holds for every plane offset and pitch residue; no read goes past the
    halo rows below the tile (one granule: 2V rows for tiles of 128 rows or
    more, else V), and the lanes store every chunk of the tile exactly once."""
    V, MC = 8, 16
    G = 2 * V if MR >= 16 else V
    for s0 in range(G):
        for L in range(G):
            reads, max_row, stored = BM.gather_reads(V, MR, MC, NT, s0, L)
            assert max_row < V * MR + G
            worst = max(BM.conflict_degree(addrs, width=2) for addrs in reads)
            assert worst == (2 if MR >= 16 else 1), (s0, L)
            want = {(C, cl, A) for C in range(MC) for cl in range(V) for A in range(MR)}
            assert len(stored) == len(want) and set(stored) == want


def test_same_gather_for_fp32_would_also_be_conflict_free_on_64_row_tiles():
    # fp32 keeps the register window (faster there), but the 8-chunk lane map
    # itself is conflict-free for 4-byte elements too
    for s0 in range(4):
        for L in range(4):
            reads, max_row, _ = BM.gather_reads(4, 8, 16, 128, s0, L)
            assert max_row < 4 * 8 + 4
            assert all(BM.conflict_degree(a, width=4) == 1 for a in reads)

