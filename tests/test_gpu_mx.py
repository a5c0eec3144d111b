"""MX scaling on the GPU (power-of-two UE8M0 scale per 32 contraction elements, applied by the
tensor cores' block scaling) against the oracle.

The GEMM: integer-valued codes with distinct exponents per row, column and group make every
output exact, so the result must equal the oracle's bit for bit (a scale byte read from the
wrong place changes it); random codes and exponents within the bound, ragged M and N, several
K blocks, every format pair. The casts: codes, scale bytes and counters bit-exact against the
oracle's MX quantise, rows grouped along x's rows and a weight grouped down its columns
(written transposed), special values and ragged shapes. The layer forward end to end, small
and at the fine-grained forward's full size on sampled rows and columns.

The scale bytes travel in the tensor cores' layout (512-byte atoms of 128 MN indices x 4
groups); the helpers below only move bytes between that layout and [MN, K/32] arrays."""
import numpy as np
import pytest
import torch

from datagen import bf16_bits_from_f32, channel_scaled_bf16, normal_bf16, workload_inputs
from oracle import fp8, gemm, quant

from gpu_util import dev_bf16, dev_u8, empty_u8, host_bf16_f64, host_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import fp8_mixed_precision_saturating_gb300 as m
    return m


def sf_size(mn, k):
    return -(-mn // 128) * (k // 128) * 512


def sf_offsets(mn, groups):
    m = np.arange(mn)[:, None]
    gg = np.arange(groups)[None, :]
    nkb = groups // 4
    return ((m // 128) * nkb + gg // 4) * 512 + 16 * (m % 32) + 4 * ((m // 32) % 4) + gg % 4


def sf_tile(e_bytes):
    """[MN, K/32] scale bytes -> the atom layout (padding rows hold 127, i.e. e = 0)."""
    mn, groups = e_bytes.shape
    out = np.full(sf_size(mn, groups * 32), 127, dtype=np.uint8)
    out[sf_offsets(mn, groups)] = e_bytes
    return out


def sf_untile(buf, mn, groups):
    return np.asarray(buf)[sf_offsets(mn, groups)]


def small_int_codes(rng, shape, fmt):
    """Codes of the values -3 .. 3 (exact products and sums)."""
    vals = rng.integers(-3, 4, size=shape).astype(np.float64)
    return fp8.cast(vals, fmt), vals


def run_mm(g, A, fa, B, fb, ea, eb, M, N, K):
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    sa = dev_u8(sf_tile((ea + 127).astype(np.uint8)))
    sb = dev_u8(sf_tile((eb + 127).astype(np.uint8)))
    g.fp8_scaled_mm(dev_u8(A), fa, dev_u8(B), fb, M, N, K, K, K, g.FP8_GRAN_MX_1x32, sa, sb, C, N)
    torch.cuda.synchronize()
    g.fp8_poll_device_error()
    return host_bf16_f64(C)


FMTS = {0: fp8.E4M3, 1: fp8.E5M2}


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (128, 128, 128), (256, 512, 512), (200, 384, 256)])
def test_mx_gemm_exact_on_integer_codes(g, M, N, K):
    """Exponents in [-4, 4] per (row, group) and (column, group), codes of -3 .. 3: each output
    is a sum of K small integers times powers of two, exact in fp32 and in bf16 here."""
    rng = np.random.default_rng(M + N + K)
    A, _ = small_int_codes(rng, (M, K), fp8.E4M3)
    B, _ = small_int_codes(rng, (N, K), fp8.E4M3)
    ea = rng.integers(-4, 5, size=(M, K // 32))
    eb = rng.integers(-4, 5, size=(N, K // 32))
    got = run_mm(g, A, 0, B, 0, ea, eb, M, N, K)
    ref, _ = gemm.mx_scaled_mm(A, fp8.E4M3, ea, B, fp8.E4M3, eb)
    assert np.array_equal(gemm.bf16_round(ref), ref)
    bad = got != ref
    assert not bad.any(), f"{bad.sum()} of {bad.size} differ; first at {np.argwhere(bad)[:4].tolist()}"


@pytest.mark.parametrize("M,N,K,fa,fb", [(300, 272, 384, 0, 0), (1024, 1280, 640, 0, 0), (129, 640, 256, 1, 0),
                                         (512, 128, 1024, 0, 1), (64, 2048, 128, 1, 1)])
def test_mx_gemm_random_against_oracle(g, M, N, K, fa, fb):
    rng = np.random.default_rng(M * 7 + N + K)
    okA = np.array([c for c in range(256) if np.isfinite(fp8.decode(c, FMTS[fa]))], dtype=np.uint8)
    okB = np.array([c for c in range(256) if np.isfinite(fp8.decode(c, FMTS[fb]))], dtype=np.uint8)
    A = rng.choice(okA, size=(M, K))
    B = rng.choice(okB, size=(N, K))
    ea = rng.integers(-20, 10, size=(M, K // 32))
    eb = rng.integers(-20, 10, size=(N, K // 32))
    got = run_mm(g, A, fa, B, fb, ea, eb, M, N, K)
    ref, mag = gemm.mx_scaled_mm(A, FMTS[fa], ea, B, FMTS[fb], eb)
    ok = gemm.within_bound(got, ref, mag)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside the bound"


def check_quant(got_q, got_sf, got_snap, o, mn, groups):
    assert np.array_equal(got_q, o["q"])
    assert np.array_equal(sf_untile(got_sf, mn, groups), o["ue8m0"])
    pad = np.ones(sf_size(mn, groups * 32), dtype=bool)
    pad[sf_offsets(mn, groups).ravel()] = False
    assert np.all(got_sf[pad] == 127)
    assert got_snap["overflow"] == o["overflow"] and got_snap["underflow"] == o["underflow"]
    assert np.float32(got_snap["amax_cur"]) == o["amax"].max()


def special_values(rng, shape):
    x = rng.standard_normal(shape) * 10.0 ** rng.uniform(-8, 8, size=(shape[0], shape[1] // 32)).repeat(32, axis=1)
    flat = x.reshape(-1)
    idx = rng.choice(flat.size, size=min(64, flat.size), replace=False)
    flat[idx[:8]] = np.nan
    flat[idx[8:12]] = np.inf
    flat[idx[12:16]] = -np.inf
    flat[idx[16:24]] = 0.0
    flat[idx[24:32]] = -0.0
    flat[idx[32:40]] = 1e-39     # bf16 subnormals
    x[:, :32] = 0.0              # an all-zero group (e = 0)
    x[0, 32:64] = 1e-40          # a group with a subnormal amax (e clamped)
    return bf16_bits_from_f32(x.astype(np.float32))


@pytest.mark.parametrize("rows,cols,fc", [(256, 512, 0), (200, 384, 1), (1, 128, 0), (1000, 1024, 0)])
def test_mx_quantize_rows_against_oracle(g, rows, cols, fc):
    rng = np.random.default_rng(rows + cols + fc)
    x_b = special_values(rng, (rows, cols))
    st = g.TensorState()
    q = empty_u8(rows, cols)
    sf = torch.full((sf_size(rows, cols),), 0xAB, dtype=torch.uint8, device="cuda")
    g.fp8_quantize(dev_bf16(x_b), rows, cols, cols, fc, g.FP8_GRAN_MX_1x32, g.FP8_SCALE_CURRENT, st, q, None, sf)
    torch.cuda.synchronize()
    o = quant.quantize_mx(x_b, FMTS[fc])
    check_quant(host_u8(q), host_u8(sf), st.snapshot(), o, rows, cols // 32)


@pytest.mark.parametrize("K,N,fc", [(256, 512, 0), (384, 200, 0), (128, 136, 1), (1024, 1000, 0)])
def test_mx_quantize_columns_transposed_against_oracle(g, K, N, fc):
    """A weight W [K, N]: groups of 32 down each column (along K), codes written as W_q^T."""
    rng = np.random.default_rng(K * 3 + N + fc)
    w_b = special_values(rng, (N, K)).T.copy()   # groups of W's columns carry the special values
    st = g.TensorState()
    qT = empty_u8(N, K)
    sf = torch.full((sf_size(N, K),), 0xAB, dtype=torch.uint8, device="cuda")
    g.fp8_quantize(dev_bf16(w_b), K, N, N, fc, g.FP8_GRAN_MX_1x32, g.FP8_SCALE_CURRENT, st, None, qT, sf)
    torch.cuda.synchronize()
    o = quant.quantize_mx(np.ascontiguousarray(w_b.T), FMTS[fc])
    check_quant(host_u8(qT), host_u8(sf), st.snapshot(), o, N, K // 32)


def test_mx_rejections(g):
    x = torch.zeros(128, 200, dtype=torch.bfloat16, device="cuda")
    q = empty_u8(128, 200)
    sf = empty_u8(4096)
    with pytest.raises(g.Fp8Error) as e:  # contraction not a multiple of 128
        g.fp8_quantize(x, 128, 200, 200, 0, g.FP8_GRAN_MX_1x32, g.FP8_SCALE_CURRENT, None, q, None, sf)
    assert e.value.status == g.FP8_ERR_UNSUPPORTED
    with pytest.raises(g.Fp8Error) as e:  # both outputs
        g.fp8_quantize(x, 128, 128, 200, 0, g.FP8_GRAN_MX_1x32, g.FP8_SCALE_CURRENT, None, q, q, sf)
    assert e.value.status == g.FP8_ERR_INVALID_ARG
    with pytest.raises(g.Fp8Error) as e:  # delayed scaling
        g.fp8_quantize(x, 128, 128, 200, 0, g.FP8_GRAN_MX_1x32, g.FP8_SCALE_DELAYED, g.TensorState(), q, None, sf)
    assert e.value.status == g.FP8_ERR_UNSUPPORTED
    C = torch.empty(128, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.Fp8Error) as e:  # K not a multiple of 128
        g.fp8_scaled_mm(q, 0, q, 0, 128, 128, 64, 64, 64, g.FP8_GRAN_MX_1x32, sf, sf, C, 128)
    assert e.value.status == g.FP8_ERR_UNSUPPORTED


def mx_forward(g, x_b, w_b, M, K, N):
    x, w = dev_bf16(x_b), dev_bf16(w_b)
    wqT, xq = empty_u8(N, K), empty_u8(M, K)
    wsf, xsf = empty_u8(sf_size(N, K)), empty_u8(sf_size(M, K))
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    X = g.FP8_GRAN_MX_1x32
    g.fp8_requantize_weights(w, K, N, X, g.FP8_SCALE_CURRENT, None, None, wqT, wsf)
    g.fp8_linear_fwd(x, M, K, N, wqT, None, wsf, None, X, g.FP8_SCALE_CURRENT, xq, None, xsf, y)
    torch.cuda.synchronize()
    g.fp8_poll_device_error()
    return y, xq, xsf, wqT, wsf


@pytest.mark.parametrize("M,K,N", [(256, 512, 768), (100, 256, 384)])
def test_mx_forward_small_against_oracle(g, M, K, N):
    x_b = channel_scaled_bf16(8100 + M, (M, K))
    w_b = normal_bf16(8101 + M, (K, N), 0.02)
    y, xq, xsf, wqT, wsf = mx_forward(g, x_b, w_b, M, K, N)
    ox = quant.quantize_mx(x_b, fp8.E4M3)
    ow = quant.quantize_mx(np.ascontiguousarray(w_b.T), fp8.E4M3)
    assert np.array_equal(host_u8(xq), ox["q"]) and np.array_equal(host_u8(wqT), ow["q"])
    assert np.array_equal(sf_untile(host_u8(xsf), M, K // 32), ox["ue8m0"])
    assert np.array_equal(sf_untile(host_u8(wsf), N, K // 32), ow["ue8m0"])
    ref, mag = gemm.mx_scaled_mm(ox["q"], fp8.E4M3, ox["e"], ow["q"], fp8.E4M3, ow["e"])
    ok = gemm.within_bound(host_bf16_f64(y), ref, mag)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside the bound"


@pytest.mark.slow
def test_mx_forward_full_size_sampled(g):
    """The fine-grained forward's full size (x [16384 x 4096], W [4096 x 14336]) with MX scales:
    64 sampled rows of x and 64 sampled columns of W quantised by the oracle (codes and scale
    bytes compared), and the 4096 outputs they meet against the exact sampled reference."""
    w_in = workload_inputs("finegrained_fwd")
    M, K, N = w_in["M"], w_in["K"], w_in["N"]
    y, xq, xsf, wqT, wsf = mx_forward(g, w_in["x"], w_in["w"], M, K, N)
    rng = np.random.default_rng(44)
    rs = np.sort(rng.choice(M, 64, replace=False))
    cs = np.sort(rng.choice(N, 64, replace=False))
    ox = quant.quantize_mx(w_in["x"][rs], fp8.E4M3)
    ow = quant.quantize_mx(np.ascontiguousarray(w_in["w"][:, cs].T), fp8.E4M3)
    assert np.array_equal(host_u8(xq)[rs], ox["q"]) and np.array_equal(host_u8(wqT)[cs], ow["q"])
    assert np.array_equal(sf_untile(host_u8(xsf), M, K // 32)[rs], ox["ue8m0"])
    assert np.array_equal(sf_untile(host_u8(wsf), N, K // 32)[cs], ow["ue8m0"])
    ii, jj = np.meshgrid(np.arange(64), np.arange(64), indexing="ij")
    ii, jj = ii.ravel(), jj.ravel()
    ref, mag = gemm.mx_scaled_mm_sampled(ox["q"], fp8.E4M3, ox["e"], ow["q"], fp8.E4M3, ow["e"], ii, jj)
    got = host_bf16_f64(y)[rs[ii], cs[jj]]
    ok = gemm.within_bound(got, ref, mag)
    assert ok.all(), f"{(~ok).sum()} of {ok.size} outside the bound"
