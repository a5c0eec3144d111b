"""GPU parity of fp8_update_requantize_weights (the optimizer step's update fused with the
weight-cache refresh) against the oracle: the updated bf16 master weight, the E4M3 codes
(row-major and transposed) and the scaling state bit for bit."""
import numpy as np
import pytest
import torch

from datagen import normal_bf16, perturbation_f32
from oracle import fp8, linear, quant

from gpu_util import dev_bf16, empty_u8, host_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import fp8_mixed_precision_saturating_gb300 as m
    return m


def host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("K,N", [(256, 384), (144, 200), (1536, 6144)])
def test_update_requantize_current(g, K, N):
    w = normal_bf16(K + N, (K, N), 0.02)
    delta = perturbation_f32(K * 7 + N, (K, N), 1e-3)
    wd = dev_bf16(w)
    st = g.TensorState()
    wq, wqT = empty_u8(K, N), empty_u8(N, K)
    g.fp8_update_requantize_weights(wd, torch.from_numpy(delta).cuda(), K, N, g.FP8_SCALE_CURRENT, st, wq, wqT)
    torch.cuda.synchronize()
    w2 = linear.perturb_master(w, delta)
    assert np.array_equal(host_bits(wd), w2)
    ref = quant.quantize_tensor(w2, fp8.E4M3)
    assert np.array_equal(host_u8(wq), ref["q"]) and np.array_equal(host_u8(wqT), ref["qT"])
    snap = st.snapshot()
    assert np.float32(snap["amax_cur"]) == ref["amax"] and np.float32(snap["scale"]) == ref["s"]
    assert np.float32(snap["scale_inv"]) == ref["d"]
    assert snap["overflow"] == ref["overflow"] and snap["underflow"] == ref["underflow"]


def test_update_requantize_delayed_trajectory(g):
    K, N, H, T = 256, 512, 4, 12
    w = normal_bf16(901, (K, N), 0.02)
    wd = dev_bf16(w)
    st = g.TensorState(hist_len=H)
    ost = quant.DelayedState(H)
    wq, wqT = empty_u8(K, N), empty_u8(N, K)
    for t in range(T):
        delta = perturbation_f32(902 + t, (K, N), 3e-3)  # large enough to grow past the history
        g.fp8_update_requantize_weights(wd, torch.from_numpy(delta).cuda(), K, N, g.FP8_SCALE_DELAYED, st, wq, wqT)
        g.fp8_history_commit(st)
        w = linear.perturb_master(w, delta)
        ref = ost.quantize(w, fp8.E4M3)
        ost.commit()
        assert np.array_equal(host_bits(wd), w), t
        assert np.array_equal(host_u8(wq), ref["q"]) and np.array_equal(host_u8(wqT), ref["qT"]), t
        a, b = st.snapshot(), ost.snapshot()
        assert a["count"] == b["count"] and np.array_equal(a["hist"], b["hist"])
        assert np.float32(a["scale"]) == b["scale"] and np.float32(a["amax_cur"]) == b["amax_cur"]
        assert a["overflow"] == b["overflow"] and a["underflow"] == b["underflow"]
    assert ost.overflow > 0  # the growing weight saturated against its history at some step


def test_update_requantize_rejections(g):
    st = g.TensorState()
    w = dev_bf16(normal_bf16(1, (16, 16)))
    d = torch.zeros(16, 16, device="cuda")
    q = empty_u8(16, 16)
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_update_requantize_weights(w, d, 16, 12, g.FP8_SCALE_CURRENT, st, q, None)
    assert e.value.status == g.FP8_ERR_UNSUPPORTED
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_update_requantize_weights(w, None, 16, 16, g.FP8_SCALE_CURRENT, st, q, None)
    assert e.value.status == g.FP8_ERR_INVALID_ARG
