"""Sizes past 2**31 elements and 2**32 bytes: 64-bit index arithmetic in every
kernel.  The oracle cannot run at this size in seconds, so the checks are the
definition at sampled positions and a permutation invariant over all of it."""
import pytest

from shared_memory_tiled_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from shared_memory_tiled_gb300 import build
    build.build()
    B.load()


def _sampled_check(x, out, rows, cols, ld_in, ld_out, n=1 << 16, seed=0):
    import torch
    g = torch.Generator(device="cuda").manual_seed(seed)
    i = torch.randint(0, rows, (n,), device="cuda", generator=g)
    j = torch.randint(0, cols, (n,), device="cuda", generator=g)
    # include the last row and column explicitly
    i = torch.cat([i, torch.tensor([rows - 1, rows - 1, 0], device="cuda")])
    j = torch.cat([j, torch.tensor([cols - 1, 0, cols - 1], device="cuda")])
    assert torch.equal(out[j * ld_out + i], x[i * ld_in + j])


@pytest.mark.parametrize("variant,schedule", [(B.Variant.AUTO, 0), (B.Variant.TMA, 0),
                                              (B.Variant.TMA, 3), (B.Variant.TMA, 4)])
def test_fp32_beyond_2_31_elements(variant, schedule):
    import torch
    rows, cols = 65537, 32801          # 2,149,679,137 elements, 8.6 GB each way
    ld_in, ld_out = 32804, 65540       # 16-byte aligned pitches (TMA-eligible)
    x = torch.randint(-2**31, 2**31 - 1, (rows * ld_in,), dtype=torch.int32, device="cuda")
    out = torch.zeros(cols * ld_out, dtype=torch.int32, device="cuda")
    args = B.make_args(x.data_ptr(), out.data_ptr(), B.DType.F32, 1, rows, cols, ld_in, ld_out)
    B.check(B.tr_transpose_ex(args, B.make_options(variant, schedule=schedule)))
    torch.cuda.synchronize()
    _sampled_check(x, out, rows, cols, ld_in, ld_out)
    # permutation invariant: the logical elements' sum (as int64) is unchanged
    xs = x.view(rows, ld_in)[:, :cols].to(torch.int64).sum()
    os_ = out.view(cols, ld_out)[:, :rows].to(torch.int64).sum()
    assert int(xs) == int(os_)
    del x, out
    torch.cuda.empty_cache()


def test_bf16_batched_beyond_2_32_bytes():
    import torch
    batch, rows, cols = 3, 40000, 24000   # 2.88e9 elements, 5.76 GB each way
    x = torch.randint(-2**15, 2**15 - 1, (batch * rows * cols,), dtype=torch.int16, device="cuda")
    out = torch.zeros_like(x)
    B.check(B.tr_transpose_batched_bf16(x.data_ptr(), out.data_ptr(), batch, rows, cols, cols,
                                        rows, rows * cols, rows * cols))
    torch.cuda.synchronize()
    xv = x.view(batch, rows, cols)
    ov = out.view(batch, cols, rows)
    g = torch.Generator(device="cuda").manual_seed(1)
    b = torch.randint(0, batch, (1 << 16,), device="cuda", generator=g)
    i = torch.randint(0, rows, (1 << 16,), device="cuda", generator=g)
    j = torch.randint(0, cols, (1 << 16,), device="cuda", generator=g)
    assert torch.equal(ov[b, j, i], xv[b, i, j])
    assert torch.equal(ov[-1, -1, :], xv[-1, :, -1])
    del x, out
    torch.cuda.empty_cache()


def test_inplace_beyond_2_31_elements():
    import torch
    n = 46349                              # 2,148,229,801 elements
    x = torch.randint(-2**31, 2**31 - 1, (n * n,), dtype=torch.int32, device="cuda")
    ref = x.view(n, n)[:4096, :4096].clone(), x.view(n, n)[-3:, :].clone()
    B.check(B.tr_transpose_inplace_f32(x.data_ptr(), 1, n, n, n * n))
    torch.cuda.synchronize()
    v = x.view(n, n)
    assert torch.equal(v[:4096, :4096], ref[0].t())
    assert torch.equal(v[:, -3:], ref[1].t())
    del x
    torch.cuda.empty_cache()


@pytest.mark.parametrize("ld_in,ld_out", [(32804, 65539), (32803, 65540)],
                         ids=["odd-output-pitch", "odd-input-pitch"])
def test_fp32_misaligned_pitches_beyond_2_31_elements(ld_in, ld_out):
    """Past 2**31 elements with rows that start off 16-byte boundaries: the
    shifted stores (with their halo rows) on the output side, per-chunk 4-byte
    loads on the input side."""
    import torch
    rows, cols = 65537, 32801          # 2,149,679,137 elements
    x = torch.randint(-2**31, 2**31 - 1, (rows * ld_in,), dtype=torch.int32, device="cuda")
    out = torch.zeros(cols * ld_out, dtype=torch.int32, device="cuda")
    args = B.make_args(x.data_ptr(), out.data_ptr(), B.DType.F32, 1, rows, cols, ld_in, ld_out)
    B.check(B.tr_transpose_ex(args, B.make_options(B.Variant.AUTO)))
    torch.cuda.synchronize()
    _sampled_check(x, out, rows, cols, ld_in, ld_out, seed=3)
    # every output row ends where it should: the element after it (pitch padding) is untouched
    pad = out.view(cols, ld_out)[:, rows:]
    assert int(torch.count_nonzero(pad)) == 0
    xs = x.view(rows, ld_in)[:, :cols].to(torch.int64).sum()
    os_ = out.view(cols, ld_out)[:, :rows].to(torch.int64).sum()
    assert int(xs) == int(os_)
    del x, out, pad
    torch.cuda.empty_cache()


@pytest.mark.parametrize("ld_in,ld_out", [(32803, 65544), (32803, 65539)],
                         ids=["odd-input-pitch", "both-pitches-odd"])
def test_bf16_misaligned_pitches_beyond_2_31_elements(ld_in, ld_out):
    """bf16 past 2**31 elements with input rows at every 2-byte offset from a
    16-byte boundary: aligned chunks realigned on chip (row offsets taken from
    the low 32 bits of the addresses), alone and with shifted stores."""
    import torch
    rows, cols = 65537, 32801          # 2,149,679,137 elements, 4.3 GB each way
    x = torch.randint(-2**15, 2**15 - 1, (rows * ld_in,), dtype=torch.int16, device="cuda")
    out = torch.zeros(cols * ld_out, dtype=torch.int16, device="cuda")
    args = B.make_args(x.data_ptr(), out.data_ptr(), B.DType.BF16, 1, rows, cols, ld_in, ld_out)
    B.check(B.tr_transpose_ex(args, B.make_options(B.Variant.AUTO)))
    torch.cuda.synchronize()
    _sampled_check(x, out, rows, cols, ld_in, ld_out, seed=5)
    pad = out.view(cols, ld_out)[:, rows:]
    assert int(torch.count_nonzero(pad)) == 0
    xs = x.view(rows, ld_in)[:, :cols].to(torch.int64).sum()
    os_ = out.view(cols, ld_out)[:, :rows].to(torch.int64).sum()
    assert int(xs) == int(os_)
    del x, out, pad
    torch.cuda.empty_cache()
