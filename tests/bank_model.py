"""Host-side model of shared-memory banking, and the address each lane of a warp
produces in every shared-memory access of the transpose kernels.

Bank model ("Shared memory and the bank conflict", section "Banks";
"Shared-memory tiling and bank conflicts", "Calculate the bank mapping"): 32
banks, successive 4-byte words in successive banks, so word w lives in bank
w mod 32.  Lanes reading the same word are served together (broadcast,
"Shared Memory and Bank Conflicts", "how banking works"); different words in
one bank are served one after another, so an n-way conflict costs n passes.

Accesses wider than 4 bytes are served in phases: a 16-byte access by a warp
is served 8 lanes at a time (each lane covers 4 consecutive banks), so the
minimum is 4 passes per warp instruction.  The model counts passes the same
way: per phase, the largest number of distinct words any bank must deliver.

The per-kernel address functions restate the index arithmetic of the CUDA
kernels so their conflict degree can be computed here, on the CPU, and then
compared with the counters Nsight Compute reports on the GPU.  The model
covers one warp instruction on its own.  Nsight's conflict counter also
charges an LSU access for cycles it waits while the TMA unit reads or writes
the same banks (a kernel rebuilt without its TMA box loads and stores reads
0-3% extra wavefronts, and up to 71% with them), and the bf16 in-place kernel
for cycles lost while other warps' global loads return; the model predicts
neither.
"""
from __future__ import annotations

from collections import defaultdict

BANKS = 32
WORD = 4


def passes(byte_addrs, width=4):
    """Shared-memory passes for one warp instruction in which lane i accesses
    ``width`` bytes at ``byte_addrs[i]`` (None = inactive lane)."""
    lanes_per_phase = {2: 32, 4: 32, 8: 16, 16: 8}[width]
    total = 0
    for p0 in range(0, 32, lanes_per_phase):
        words_in_bank = defaultdict(set)
        for a in byte_addrs[p0:p0 + lanes_per_phase]:
            if a is None:
                continue
            for w in range(a // WORD, max(a // WORD + 1, (a + width) // WORD)):
                words_in_bank[w % BANKS].add(w)
        total += max((len(s) for s in words_in_bank.values()), default=0)
    return total


def conflict_degree(byte_addrs, width=4):
    """Passes divided by the conflict-free minimum (1 = conflict-free)."""
    minimum = {2: 1, 4: 1, 8: 2, 16: 4}[width]
    return passes(byte_addrs, width) / minimum


# --- the page's 32 x (32+pad) tile, 4-byte elements -------------------------------------

def pad_tile_column_read(pad, col=0, esize=4):
    """Phase-2 read of the padded tile: lane t reads tile[t][col]."""
    return [(t * (32 + pad) + col) * esize for t in range(32)]


def pad_tile_row_write(pad, row=0, esize=4):
    """Phase-1 write: lane t writes tile[row][t]."""
    return [(row * (32 + pad) + t) * esize for t in range(32)]


# --- the vectorised swizzled tile (tile_vec.cu) ------------------------------------------

def vec_tile_load_store(warp, k, V=4, MC=16):
    """Phase-1 16-byte store of load k: thread t holds chunk t % MC of tile row
    t // MC + k * 256 // MC, stored at chunk position cc ^ ((r // V) % 8)."""
    out = []
    for lane in range(32):
        t = warp * 32 + lane
        cc, r = t % MC, t // MC + k * (256 // MC)
        out.append((r * MC + (cc ^ ((r // V) & 7))) * 16)
    return out


def vec_tile_read(warp, m, V=4, MR=16, MC=16, j=0):
    """Phase-2 16-byte read m of micro-block u = t + 256 j: A = u % MR, C = u // MR,
    tile row V*A + m, chunk C at position C ^ (A % 8)."""
    out = []
    for lane in range(32):
        u = warp * 32 + lane + 256 * j
        A, C = u % MR, u // MR
        out.append(((V * A + m) * MC + (C ^ (A & 7))) * 16)
    return out


def vec_tile_staging(warp, k, MC=16, next_chunk=False):
    """Misaligned input rows: thread t's aligned chunk of load k (chunk t % MC of
    tile row t // MC + k * 256 // MC) stored unshifted in staging rows of MC + 1
    chunks, or with ``next_chunk`` the read of the chunk after it."""
    out = []
    for lane in range(32):
        t = warp * 32 + lane
        cc, r = t % MC, t // MC + k * (256 // MC)
        out.append((r * (MC + 1) + cc + int(next_chunk)) * 16)
    return out


def vec_tile_staging_helper(warp, TR, MC=16):
    """The helper store: thread t puts the chunk past tile row t at position MC
    of that row's staging row (threads t >= TR hold none)."""
    out = []
    for lane in range(32):
        rr = warp * 32 + lane
        out.append((rr * (MC + 1) + MC) * 16 if rr < TR else None)
    return out


# --- the TMA tile with the 128-byte hardware swizzle (tile_tma.cu) ------------------------

def _tma_lane(warp, lane):
    quad = warp >> 1
    s = (lane >> 3) + 4 * (warp & 1)
    c = lane & 7
    a = c ^ s
    return 8 * (quad >> 1) + a, 8 * (quad & 1) + c, a, c


def tma_read(warp, m, V=4):
    """LSU read m of the TMA input box: row V*A+m, chunk c at c ^ (row % 8)."""
    box = 16 * V * 128
    out = []
    for lane in range(32):
        A, C, a, c = _tma_lane(warp, lane)
        r = V * A + m
        out.append((C >> 3) * box + r * 128 + ((c ^ (r & 7)) << 4))
    return out


def tma_write(warp, m, V=4):
    """LSU write m into the TMA output box: row V*C+m, chunk a at a ^ (row % 8)."""
    box = 16 * V * 128
    out = []
    for lane in range(32):
        A, C, a, c = _tma_lane(warp, lane)
        o = V * C + m
        out.append((A >> 3) * box + o * 128 + ((a ^ (o & 7)) << 4))
    return out


def ws_consumer_read(warp, m, V=4):
    """Warp-specialised pipeline (k_tma_ws), consumer read m: thread t < 256 owns
    micro-block (A, C) = (t % 16, t // 16) and reads tile row V*A + (m + rot) % V
    with rot = (A // 2) % 4 (fp32) or A % 8 (bf16), chunk C of the two-box slot."""
    box = 16 * V * 128
    out = []
    for lane in range(32):
        t = warp * 32 + lane
        A, C = t & 15, t >> 4
        rot = ((A >> 1) & 3) if V == 4 else (A & 7)
        r = V * A + ((m + rot) & (V - 1))
        out.append((C >> 3) * box + r * 128 + (((C & 7) ^ (r & 7)) << 4))
    return out


def ldst_read(m, p, V=4):
    """Per-warp load-only pipeline (k_tma_ldst), read m of pass p: lane owns
    A = lane % 8, C = 4p + lane // 8 in one 8V-row box, row V*A + (m + rot) % V
    with rot = A // 2 (fp32) or A (bf16)."""
    out = []
    for lane in range(32):
        A = lane & 7
        rot = (A >> 1) if V == 4 else A
        C = 4 * p + (lane >> 3)
        r = V * A + ((m + rot) & (V - 1))
        out.append(r * 128 + ((C ^ (r & 7)) << 4))
    return out


# --- the transposed operand store of the padded SGEMM page --------------------------------

def sgemm_as_store(BK, a_stride, j, offset=0):
    """Lane t of the first warp stores element j of its float4 of A, transposed:
    innerRowA = t // (BK/4), innerColA = t % (BK/4), word
    (innerColA*4 + j) * a_stride + innerRowA + offset ("Padded Shared Memory:
    Eliminating Bank Conflicts", section "How Shared Memory Is Addressed")."""
    out = []
    for t in range(32):
        row, col = t // (BK // 4), t % (BK // 4)
        out.append(((col * 4 + j) * a_stride + row + offset) * WORD)
    return out


def a_stride(BM, BK):
    """The page's padding rule: BM + (32 / BK) % 8 ("The Fix Is One Constant")."""
    return BM + (32 // BK) % 8


# --- the bf16 shifted stores' column gather (tile_vec_kernel.cuh) -------------------------

def gather_reads(V, MR, MC, NT, s0, L):
    """Byte addresses of the column gather's shared reads, one list of 32 per
    warp instruction: warp w, step j, element q.  Lane (k = lane % KL, a =
    (lane / KL) % RUN) of step `step` reads input row V*A + d + q of column
    V*C + cl of the swizzled tile (row pitch MC chunks, chunk cc of row r at
    position cc ^ ((r / V) % 8)), RUN being the consecutive chunks A of one
    output row an instruction covers (16 when the tile has them, else 8), KL =
    32 / RUN its output rows, cl = (V / KL) k + par, with C, the parity par and
    the run taken from the step and d the output row's offset to its next
    granule boundary, fixed by the plane offset s0 and the pitch residue L
    (both modulo the shift granule G: 2V elements, 32 bytes, for tiles of 128
    rows or more, else V).  Also returns the largest tile row read and the
    (C, cl, A) chunks stored, one entry per lane and step."""
    esize = 16 // V
    RUN = 16 if MR >= 16 else 8
    KL = 32 // RUN
    PAR, ABLK = V // KL, MR // RUN
    G = 2 * V if V * MR >= 128 else V   # shift granule
    steps = MC * PAR * ABLK
    out, max_row, stored = [], 0, []
    for w in range(NT // 32):
        for j in range(steps // (NT // 32)):
            step = w + (NT // 32) * j
            C, par, blk = step // (PAR * ABLK), (step // ABLK) % PAR, step % ABLK
            for q in range(V):
                addrs = []
                for lane in range(32):
                    k, a = lane % KL, (lane // KL) % RUN
                    cl, A = PAR * k + par, blk * RUN + a
                    d = (G - (s0 + (V * C + cl) * L) % G) % G
                    r = V * A + d + q
                    max_row = max(max_row, r)
                    addrs.append(((r * MC + (C ^ ((r // V) & 7))) * V + cl) * esize)
                    if q == 0:
                        stored.append((C, cl, A))
                out.append(addrs)
    return out, max_row, stored
