"""fp8_scaled_mm_quant: the GEMM epilogue that also emits FP8 codes of its output.

Bit-exact against the oracle on integer-valued products (every output is an integer below
256 in magnitude, so the bf16 output is exact and the oracle quantises the same values
independently): codes, amax, scale and counters with a delayed history (the fused epilogue)
and with an empty history (the bootstrap cast). At the delayed loop's forward shape
(32768 x 6144, contraction 1536) on its real operands: the codes, amax, scales and counters
against the oracle's delayed quantise of the kernel's own bf16 output (bootstrap, fused, and
fused with a history that saturates), the bf16 output on sampled entries against the exact
reference. On random data the fused codes and state also equal fp8_quantize of the kernel's
own bf16 output with the same delayed state."""
import numpy as np
import pytest
import torch

from datagen import normal_bf16
from oracle import fp8, gemm, quant

from gpu_util import dev_u8, empty_u8, host_u8, host_bf16_f64

pytestmark = pytest.mark.gpu
SMALL_INT_CODES = np.array([0xC0, 0xB8, 0x00, 0x38, 0x40], dtype=np.uint8)  # E4M3 -2, -1, 0, 1, 2


@pytest.fixture(scope="module")
def g():
    import fp8_mixed_precision_saturating_gb300 as m
    return m


def one(v):
    return torch.tensor([v], dtype=torch.float32, device="cuda")


def bf16_bits_of_exact(c):
    """bf16 bit patterns of values that bf16 represents exactly."""
    f = np.asarray(c, dtype=np.float32)
    assert np.array_equal(f.astype(np.float64), c)
    bits = f.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0)
    return (bits >> 16).astype(np.uint16)


def run(g, A, B, fc, st, M, N, K):
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    Cq = empty_u8(M, N)
    g.fp8_scaled_mm_quant(dev_u8(A), 0, dev_u8(B), 0, M, N, K, K, K, one(1.0), one(1.0), C, N, fc, st, Cq)
    torch.cuda.synchronize()
    g.fp8_poll_device_error()
    return C, Cq


@pytest.mark.parametrize("M,N,K", [(300, 272, 64), (4096, 3072, 64), (8192, 768, 32)])
@pytest.mark.parametrize("fc,fmt", [(0, fp8.E4M3), (1, fp8.E5M2)])
def test_fused_and_bootstrap_against_oracle(g, M, N, K, fc, fmt):
    rng = np.random.default_rng(M + N + K + fc)
    A = rng.choice(SMALL_INT_CODES, size=(M, K))
    B = rng.choice(SMALL_INT_CODES, size=(N, K))
    ref, _, _ = gemm.scaled_mm(A, fp8.E4M3, B, fp8.E4M3, 1.0, 1.0)
    cbits = bf16_bits_of_exact(ref)
    for hist in ([], [37.5], [3.0, 100.0, 9.0]):  # empty history = bootstrap; 37.5 saturates the tails
        st = g.TensorState(hist_len=4)
        ost = quant.DelayedState(4)
        for i, a in enumerate(hist):
            st.amax_history[i] = a
            ost.hist[i] = np.float32(a)
        st.hist_count[0] = len(hist)
        ost.count = len(hist)
        C, Cq = run(g, A, B, fc, st, M, N, K)
        assert np.array_equal(host_bf16_f64(C), ref)
        o = ost.quantize(cbits, fmt, delayed=True)
        assert np.array_equal(host_u8(Cq), o["q"]), hist
        snap = st.snapshot()
        assert np.float32(snap["amax_cur"]) == o["amax"]
        assert np.float32(snap["scale"]) == o["s"] and np.float32(snap["scale_inv"]) == o["d"]
        assert snap["overflow"] == o["overflow"] and snap["underflow"] == o["underflow"]
        assert snap["count"] == len(hist)  # the call does not push; fp8_history_commit does


def test_fused_codes_equal_the_standalone_quantiser_on_random_data(g):
    rng = np.random.default_rng(7)
    M, N, K = 2048, 1536, 512
    A = fp8.cast(rng.standard_normal((M, K)) * 20, fp8.E4M3)
    B = fp8.cast(rng.standard_normal((N, K)) * 20, fp8.E4M3)
    for fc in (0, 1):
        st1, st2 = g.TensorState(hist_len=2), g.TensorState(hist_len=2)
        for st in (st1, st2):
            st.amax_history[0] = 3.0e4
            st.hist_count[0] = 1
        C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        Cq = empty_u8(M, N)
        g.fp8_scaled_mm_quant(dev_u8(A), 0, dev_u8(B), 0, M, N, K, K, K, one(0.5), one(0.25), C, N, fc, st1, Cq)
        q2 = empty_u8(M, N)
        g.fp8_quantize(C, M, N, N, fc, g.FP8_GRAN_TENSOR, g.FP8_SCALE_DELAYED, st2, q2)
        torch.cuda.synchronize()
        assert torch.equal(Cq, q2)
        a, b = st1.snapshot(), st2.snapshot()
        for k in ("amax_cur", "scale", "scale_inv", "overflow", "underflow"):
            assert a[k] == b[k], k


def test_fused_rejections(g):
    st = g.TensorState()
    A = torch.zeros(16, 32, dtype=torch.uint8, device="cuda")
    C = torch.zeros(16, 24, dtype=torch.bfloat16, device="cuda")
    Cq = empty_u8(16, 24)
    with pytest.raises(g.Fp8Error) as e:  # N must be a multiple of 16
        g.fp8_scaled_mm_quant(A, 0, A, 0, 16, 24, 32, 32, 32, one(1.0), one(1.0), C, 24, 0, st, Cq)
    assert e.value.status == g.FP8_ERR_ALIGNMENT


def same_quant(snap, o, count):
    assert np.float32(snap["amax_cur"]) == o["amax"]
    assert np.float32(snap["scale"]) == o["s"] and np.float32(snap["scale_inv"]) == o["d"]
    assert snap["count"] == count


@pytest.mark.slow
def test_fused_epilogue_against_oracle_at_the_loop_forward_shape(g):
    """The delayed loop's forward: x [32768 x 1536] and W [1536 x 6144] (their seeds) cast per
    tensor to E4M3 by the oracle, the GEMM's output cast to E4M3 in its epilogue."""
    M, K, N = 32768, 1536, 6144
    ox = quant.quantize_tensor(normal_bf16(5000, (M, K)), fp8.E4M3)
    ow = quant.quantize_tensor(normal_bf16(5100, (K, N), 0.02), fp8.E4M3)
    A, B = dev_u8(ox["q"]), dev_u8(ow["qT"])
    da, db = one(ox["d"]), one(ow["d"])
    st, ost = g.TensorState(hist_len=16), quant.DelayedState(16)

    def call():
        C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        Cq = empty_u8(M, N)
        g.fp8_scaled_mm_quant(A, 0, B, 0, M, N, K, K, K, da, db, C, N, 0, st, Cq)
        torch.cuda.synchronize()
        g.fp8_poll_device_error()
        return C, Cq

    # 1. bootstrap (empty history): the output is cast from its own amax
    C, Cq = call()
    cbits = C.view(torch.int16).cpu().numpy().view(np.uint16)
    rng = np.random.default_rng(17)
    r, c = rng.integers(0, M, 4096), rng.integers(0, N, 4096)
    ref, mag = gemm.scaled_mm_sampled(ox["q"], fp8.E4M3, ow["qT"], fp8.E4M3, ox["d"], ow["d"], r, c)
    ok = gemm.within_bound(host_bf16_f64(C)[r, c], ref, mag)
    assert ok.all(), f"{(~ok).sum()} outputs outside the bound"
    o = ost.quantize(cbits, fp8.E4M3, delayed=True)
    assert np.array_equal(host_u8(Cq), o["q"])
    same_quant(st.snapshot(), o, 0)
    assert st.snapshot()["overflow"] == o["overflow"] == 0 and st.snapshot()["underflow"] == o["underflow"]
    # 2. the fused epilogue with the history [amax of step 1]: the same scale, so the same codes
    g.fp8_history_commit(st)
    ost.commit()
    C2, Cq2 = call()
    assert torch.equal(C2.view(torch.int16), C.view(torch.int16))
    o2 = ost.quantize(cbits, fp8.E4M3, delayed=True)
    assert np.array_equal(host_u8(Cq2), o2["q"])
    snap = st.snapshot()
    same_quant(snap, o2, 1)
    assert snap["overflow"] == ost.overflow and snap["underflow"] == ost.underflow
    # 3. a history whose maximum is an eighth of the output's amax: the tails saturate
    small = np.float32(o["amax"] / 8)
    st.amax_history[0] = float(small)
    ost.hist[0] = small
    C3, Cq3 = call()
    o3 = ost.quantize(cbits, fp8.E4M3, delayed=True)
    assert o3["overflow"] > 0
    assert np.array_equal(host_u8(Cq3), o3["q"])
    snap = st.snapshot()
    same_quant(snap, o3, 1)
    assert snap["overflow"] == ost.overflow and snap["underflow"] == ost.underflow
