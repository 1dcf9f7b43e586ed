"""GPU parity of rowops_layernorm_gelu with the oracle, through the C ABI.

The fp32 4096 x 768 workload in full; the bf16 65536 x {8192, 127, 4097}
workloads on reduced row counts in full and at full size (benchmark launch
configuration) on sampled rows; edge cases: NULL weight / bias, ragged and
misaligned rows, in place, constant rows, every kernel variant, guard bands.
"""
import numpy as np
import pytest
import torch

from row_wise_reduction_gb300 import rowops_layernorm_gelu, workloads
from tests import _compare as C
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, gu.requires_gpu]

W2 = workloads.WORKLOADS["layernorm_gelu_f32_4096x768"]
W5 = workloads.WORKLOADS["layernorm_gelu_bf16_65536x8192"]
W5a = workloads.WORKLOADS["layernorm_gelu_bf16_65536x127"]
W5b = workloads.WORKLOADS["layernorm_gelu_bf16_65536x4097"]


def edge(dtype, M, N, seed=11, affine=True):
    return workloads.Workload(f"edge_{dtype}_{M}x{N}", "layernorm_gelu", dtype, M, N, seed=seed, affine=affine)


def host(t):
    return None if t is None else t.float().cpu().numpy()


def check(oracle, wl, ld=None, offset=0, yoffset=None, inplace=False, use_w=True, use_b=True, eps=None):
    inp = gu.make_x(wl, ld=ld, offset=offset)
    x = inp["x"]
    w = inp.get("w") if use_w else None
    b = inp.get("b") if use_b else None
    eps = wl.eps if eps is None else eps
    xin = gu.rows_f32(x)
    if inplace:
        y, buf, inside = x, None, None
    else:
        y, buf, inside = gu.guarded_like(x, offset=offset if yoffset is None else yoffset)
    rowops_layernorm_gelu(x, w, b, eps, y)
    torch.cuda.synchronize()
    ref = oracle.layernorm_gelu(xin, host(w), host(b), eps)
    err = C.assert_ln_gelu_close(C.to_f64(y), ref, wl.dtype, what=wl.name)
    if buf is not None:
        gu.assert_guard_untouched(buf, inside)
    return err


def test_ln_gelu_f32_4096x768_full(oracle):
    check(oracle, W2)


@pytest.mark.parametrize("wl", [W5, W5a, W5b], ids=lambda w: w.name)
def test_ln_gelu_bf16_reduced_rows(oracle, wl):
    check(oracle, wl.with_shape(M=1000 if wl.N > 1000 else 4099))


@pytest.mark.parametrize("wl", [W5, W5a, W5b], ids=lambda w: w.name)
def test_ln_gelu_bf16_full_size_sampled(oracle, wl):
    """Full-size bf16 workloads (65536 rows) in the default launch
    configuration: 48 sampled rows against the oracle; on every row the output
    is finite."""
    inp = gu.make_x(wl)
    x, w, b = inp["x"], inp["w"], inp["b"]
    y = rowops_layernorm_gelu(x, w, b, wl.eps)
    torch.cuda.synchronize()
    rows = gu.sample_rows(wl.M, 48, seed=wl.N)
    ref = oracle.layernorm_gelu(gu.rows_f32(x, rows), host(w), host(b), wl.eps)
    C.assert_ln_gelu_close(C.to_f64(y[torch.as_tensor(rows, device=y.device)]), ref, "bf16", what=wl.name)
    assert torch.isfinite(y).all()
    del x, y, inp


RAGGED_N = [1, 2, 3, 5, 8, 9, 17, 31, 127, 128, 129, 767, 768, 769, 4095, 4097, 8192, 12288, 16385, 20000,
            32769, 40000]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", RAGGED_N)
def test_ln_gelu_ragged_n(oracle, dtype, N):
    check(oracle, edge(dtype, 23, N, seed=N))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,ld,offset", [(127, 127, 1), (4097, 4097, 0), (4097, 4105, 3), (768, 780, 0),
                                         (8192, 8192, 1), (40000, 40003, 1)])
def test_ln_gelu_strided_and_misaligned_rows(oracle, dtype, N, ld, offset):
    check(oracle, edge(dtype, 19, N, seed=ld), ld=ld, offset=offset)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [127, 8192, 20000])
def test_ln_gelu_x_and_y_out_of_phase(oracle, dtype, N):
    check(oracle, edge(dtype, 7, N), offset=1, yoffset=0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("use_w,use_b", [(False, False), (True, False), (False, True)])
def test_ln_gelu_null_affine(oracle, dtype, use_w, use_b):
    """NULL weight / bias act as 1 / 0."""
    check(oracle, edge(dtype, 33, 768), use_w=use_w, use_b=use_b)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [768, 8192, 40000])
def test_ln_gelu_in_place(oracle, dtype, N):
    check(oracle, edge(dtype, 9, N), inplace=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ln_gelu_constant_and_shifted_rows(oracle, dtype):
    """A constant row normalises to 0 (output GELU(b)); a row with a large
    common offset normalises like the unshifted row; eps = 0 on a
    non-constant row."""
    N = 1000
    g = torch.Generator().manual_seed(5)
    x = torch.randn(4, N, generator=g)
    x[0] = 3.5
    x[1] = x[2] + 100.0
    dt = workloads.torch_dtype(dtype)
    xt = x.to(dt).cuda()
    w = (0.5 + torch.rand(N, generator=g)).to(dt).cuda()
    b = (0.1 * torch.randn(N, generator=g)).to(dt).cuda()
    for eps in (1e-5, 0.0):
        rows = [0, 1, 2, 3] if eps > 0 else [1, 2, 3]
        xs = xt[rows].contiguous()
        y = rowops_layernorm_gelu(xs, w, b, eps)
        torch.cuda.synchronize()
        ref = oracle.layernorm_gelu(xs.float().cpu().numpy(), host(w), host(b), eps)
        C.assert_ln_gelu_close(C.to_f64(y), ref, dtype)


def test_ln_gelu_large_inputs_do_not_overflow(oracle):
    """Entries far from the mean give |z| >> 10: GELU(z) = z for large
    positive z and -0 for large negative z, never NaN."""
    N = 64
    x = torch.zeros(2, N)
    x[0, 0] = 1e4
    x[1, 0] = -1e4
    w = torch.full((N,), 40.0)
    xt, wt = x.cuda(), w.cuda()
    y = rowops_layernorm_gelu(xt, wt, None, 1e-5)
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
    ref = oracle.layernorm_gelu(x.numpy(), w.numpy(), None, 1e-5)
    # |z| reaches ~317 here, where one fp32 ulp alone is 3e-5: allow 4 ulps relative
    C.assert_ln_gelu_close(C.to_f64(y), ref, "f32", rel=2.0 ** -21)


def test_ln_gelu_deterministic():
    wl = edge("bf16", 300, 8192)
    inp = gu.make_x(wl)
    a = rowops_layernorm_gelu(inp["x"], inp["w"], inp["b"], 1e-5)
    b = rowops_layernorm_gelu(inp["x"], inp["w"], inp["b"], 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_ln_gelu_empty_is_noop():
    x = torch.empty(0, 128, device="cuda")
    y = rowops_layernorm_gelu(x, None, None, 1e-5)
    torch.cuda.synchronize()
    assert y.shape == (0, 128)


VARIANTS = [(tpr, vpt) for tpr in (16, 32, 64, 128, 256, 512, 1024) for vpt in (1, 2, 3, 4)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("tpr,vpt", VARIANTS)
@pytest.mark.parametrize("offset", [0, 1])
def test_ln_gelu_every_register_variant(oracle, monkeypatch, dtype, tpr, vpt, offset):
    """Each register-resident instantiation (aligned-row form with offset 0,
    unaligned-row form with offset 1), forced, on its largest row minus a tail."""
    vec = 4 if dtype == "f32" else 8
    N = tpr * vpt * vec - (0 if offset == 0 else 3)
    if 8 * ((N + 3) // 4 * 4) > 200 * 1024:
        pytest.skip("affine staging would not fit shared memory; the looped kernel takes this size")
    monkeypatch.setenv("ROWOPS_KERNEL", "reg")
    monkeypatch.setenv("ROWOPS_FORCE_TPR", str(tpr))
    monkeypatch.setenv("ROWOPS_FORCE_VPT", str(vpt))
    check(oracle, edge(dtype, 2 * (1024 // tpr) + 1, N, seed=tpr + vpt), offset=offset)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ctas", ["-1", "1", "3"])
def test_ln_gelu_grid_modes(oracle, monkeypatch, dtype, ctas):
    monkeypatch.setenv("ROWOPS_CTAS_PER_SM", ctas)
    check(oracle, edge(dtype, 2001, 1024))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ln_gelu_forced_looped(oracle, monkeypatch, dtype):
    monkeypatch.setenv("ROWOPS_FORCE_LOOPED", "1")
    check(oracle, edge(dtype, 41, 4097), offset=1)
    check(oracle, edge(dtype, 41, 768))


TMA_VARIANTS = [(b, v) for b in (64, 128, 256, 512) for v in (1, 2, 3, 4, 8)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("block,vpt", TMA_VARIANTS)
@pytest.mark.parametrize("full", [True, False])
def test_ln_gelu_every_tma_variant(oracle, monkeypatch, dtype, block, vpt, full):
    """Each TMA-fed row-pipeline instantiation, forced (thread-major w/b
    staging included): rows of exactly block * vpt vectors and one shorter."""
    vec = 4 if dtype == "f32" else 8
    nvec = block * vpt - (0 if full else 1)
    if nvec < 64:
        pytest.skip("the row pipeline takes rows of at least 64 vectors")
    N = nvec * vec
    es = 4 if dtype == "f32" else 2
    if 2 * block * vpt * vec * 4 + 2 * ((N * es + 127) // 128 * 128) + 128 > 226 * 1024:
        pytest.skip("w/b staging plus two row buffers exceed shared memory; another kernel takes this size")
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    monkeypatch.setenv("ROWOPS_FORCE_TPR", str(block))
    monkeypatch.setenv("ROWOPS_FORCE_VPT", str(vpt))
    monkeypatch.setenv("ROWOPS_ROWS_PER_CTA", "1")
    check(oracle, edge(dtype, 2 * 152 + 3, N, seed=block * vpt))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("tpr", [128, 256])
@pytest.mark.parametrize("vpt", [2, 4, 8])
@pytest.mark.parametrize("rows", [2, 4])
def test_ln_gelu_multi_row_groups(oracle, monkeypatch, dtype, tpr, vpt, rows):
    """Several independent row groups per CTA sharing one w/b staging, each with
    its own ring and named barrier; M not a multiple of the group count."""
    vec = 4 if dtype == "f32" else 8
    es = 4 if dtype == "f32" else 2
    N = tpr * vpt * vec
    if 2 * tpr * vpt * vec * 4 + rows * 2 * ((N * es + 127) // 128 * 128) + 128 > 226 * 1024:
        pytest.skip("does not fit shared memory; the dispatcher picks fewer row groups")
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    monkeypatch.setenv("ROWOPS_FORCE_TPR", str(tpr))
    monkeypatch.setenv("ROWOPS_FORCE_VPT", str(vpt))
    monkeypatch.setenv("ROWOPS_ROWS_PER_CTA", str(rows))
    check(oracle, edge(dtype, 152 * rows + 3, N, seed=tpr + vpt + rows))
    check(oracle, edge(dtype, 5, N, seed=7), inplace=True)
    from row_wise_reduction_gb300 import rowops_device_status

    assert rowops_device_status() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ring", ["2", "5"])
@pytest.mark.parametrize("ctas", ["0", "1", "-1"])
@pytest.mark.parametrize("use_wb", [True, False])
def test_ln_gelu_tma_ring_depths_grids_affine(oracle, monkeypatch, dtype, ring, ctas, use_wb):
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    monkeypatch.setenv("ROWOPS_RING_BUFFERS", ring)
    monkeypatch.setenv("ROWOPS_CTAS_PER_SM", ctas)
    check(oracle, edge(dtype, 700, 2048), use_w=use_wb, use_b=use_wb)
    from row_wise_reduction_gb300 import rowops_device_status

    assert rowops_device_status() == 0


def test_ln_gelu_tma_in_place_and_strided(oracle, monkeypatch):
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    check(oracle, edge("bf16", 301, 8192), inplace=True)
    check(oracle, edge("bf16", 301, 8192), ld=8192 + 64)
    check(oracle, edge("f32", 77, 768), ld=768 + 4)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,ld,offset", [(4097, 4097, 0), (8191, 8191, 0), (1000, 1003, 1), (3001, 3001, 2),
                                         (8192, 8192, 3), (12345, 12350, 1)])
@pytest.mark.parametrize("rows", ["1", "2", "4"])
def test_ln_gelu_tma_general_rows(oracle, monkeypatch, dtype, N, ld, offset, rows):
    """The row pipeline's general form: rows that start anywhere (x and y in the
    same 16-byte phase), bulk-copied aligned bodies, unaligned heads and tails
    loaded directly, w/b read from column order with the widest access each
    row's alignment allows; one, two or four row groups per CTA."""
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    monkeypatch.setenv("ROWOPS_ROWS_PER_CTA", rows)
    check(oracle, edge(dtype, 157, N, seed=N + offset), ld=ld, offset=offset)
    from row_wise_reduction_gb300 import rowops_device_status

    assert rowops_device_status() == 0


@pytest.mark.parametrize("M", [1, 3, 9])
@pytest.mark.parametrize("rows", ["1", "4"])
def test_ln_gelu_tma_fewer_rows_than_phase_classes(oracle, monkeypatch, M, rows):
    """4097-column bf16 rows start at 8 different offsets modulo 16 bytes; each
    CTA of the general row pipeline takes one such class, so with fewer rows
    than classes some CTAs have nothing to do and the rest one row each."""
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    monkeypatch.setenv("ROWOPS_ROWS_PER_CTA", rows)
    check(oracle, edge("bf16", M, 4097, seed=M))
    from row_wise_reduction_gb300 import rowops_device_status

    assert rowops_device_status() == 0


@pytest.mark.parametrize("dtype,N,ld,offset", [("bf16", 8192, 8192, 0), ("f32", 4096, 4096, 0),
                                               ("bf16", 8190, 8190, 0), ("bf16", 8192, 8200, 3)])
@pytest.mark.parametrize("M", [3, 5, 777])
def test_ln_gelu_tma_five_row_groups(oracle, monkeypatch, dtype, N, ld, offset, M):
    """Five row groups of 128 threads x 8 vectors in a 640-thread CTA (the tile
    of 8192-column bf16 and 4096-column fp32 rows): full and general rows,
    fewer rows than groups, a ragged last round."""
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    monkeypatch.setenv("ROWOPS_ROWS_PER_CTA", "5")
    check(oracle, edge(dtype, M, N, seed=M + N + offset), ld=ld, offset=offset)
    from row_wise_reduction_gb300 import rowops_device_status

    assert rowops_device_status() == 0


@pytest.mark.parametrize("dtype,M,N", [("f32", 4096, 768), ("bf16", 3000, 2048), ("f32", 300, 8192)])
def test_ln_gelu_small_batches_take_register_rows(oracle, dtype, M, N):
    """Batches of at most 32 MiB go to the register-resident kernel by
    default; the result equals the row pipeline's within the tolerance."""
    check(oracle, edge(dtype, M, N, seed=M))


FLAT_N = [1, 7, 32, 33, 64, 65, 100, 127, 128, 129, 200, 255, 256, 257]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", FLAT_N)
@pytest.mark.parametrize("M", [1, 5, 1001])
def test_ln_gelu_flat_chunks(oracle, monkeypatch, dtype, N, M):
    """The kernel for short back-to-back rows by chunks of rows, forced (so
    also on rows of whole 16-byte vectors): one row, fewer rows than a chunk,
    and a last chunk whose bytes end off a 16-byte boundary (its final
    elements moved with plain loads and stores); guard bands untouched. N =
    257 is past the kernel's widths: the forced choice falls back to the
    register rows."""
    monkeypatch.setenv("ROWOPS_KERNEL", "flat")
    check(oracle, edge(dtype, M, N, seed=N + M))
    from row_wise_reduction_gb300 import rowops_device_status

    assert rowops_device_status() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ctas", ["1", "-1"])
def test_ln_gelu_flat_many_chunks_per_cta(oracle, monkeypatch, dtype, ctas):
    """One CTA per SM: every CTA takes many chunks through its two buffers,
    each refilled once the bulk store of its previous chunk has read it; and
    one CTA per chunk."""
    monkeypatch.setenv("ROWOPS_CTAS_PER_SM", ctas)
    check(oracle, edge(dtype, 20001, 127, seed=3))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ln_gelu_flat_in_place_and_null_affine(oracle, dtype):
    """Default choice on short unaligned back-to-back rows: in place, and with
    NULL weight or bias."""
    check(oracle, edge(dtype, 3001, 127), inplace=True)
    check(oracle, edge(dtype, 301, 127, seed=2), use_w=False)
    check(oracle, edge(dtype, 301, 127, seed=3), use_b=False)
    check(oracle, edge(dtype, 301, 129, seed=4), use_w=False, use_b=False)


@pytest.mark.parametrize("dtype,M,N", [("f32", 65536, 256), ("bf16", 5000, 64), ("f32", 3000, 128),
                                       ("bf16", 65536, 127)])
def test_ln_gelu_flat_default_choices(oracle, dtype, M, N):
    """Shapes the chunked kernel takes by default: a batch above 32 MiB of
    256-column fp32 rows, rows of at most 128 columns, and the 127-column bf16
    tail at full size, each compared in full."""
    check(oracle, edge(dtype, M, N, seed=M + N))
