"""GPU parity of the quantisers against the CPU oracle: codes, amax, scales and counters
bit-exact, through the C ABI."""
import numpy as np
import pytest
import torch

from datagen import bf16_bits_from_f32, normal_bf16, outlier_normal_bf16, lognormal_grad_bf16, channel_scaled_bf16
from oracle import fp8, quant

from gpu_util import dev_bf16, empty_u8, host_u8

pytestmark = pytest.mark.gpu

FMTS = [(0, fp8.E4M3), (1, fp8.E5M2)]


@pytest.fixture(scope="module")
def g():
    import fp8_mixed_precision_saturating_gb300 as m
    return m


def all_bf16_patterns():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 128)


def f32(t):
    return np.float32(t.item())


def check_state_tensor(st, ref, fmtname, overflow=None, underflow=None):
    s = st.snapshot()
    assert np.float32(s["amax_cur"]) == ref["amax"]
    assert np.float32(s["scale"]) == ref["s"], (s["scale"], ref["s"])
    assert np.float32(s["scale_inv"]) == ref["d"]
    if overflow is not None:
        assert s["overflow"] == overflow and s["underflow"] == underflow


@pytest.mark.parametrize("fi,fmt", FMTS)
def test_every_bf16_pattern_scale_one(g, fi, fmt):
    """All 65,536 bf16 patterns; +-inf are among them, so amax is not finite and s = 1."""
    x = all_bf16_patterns()
    xd = dev_bf16(x)
    st = g.TensorState()
    q = empty_u8(512, 128)
    g.fp8_quantize(xd, 512, 128, 128, fi, g.FP8_GRAN_TENSOR, g.FP8_SCALE_CURRENT, st, q)
    ref = quant.quantize_tensor(x, fmt)
    assert ref["s"] == 1.0
    got = host_u8(q)
    bad = np.nonzero(got != ref["q"])
    assert got.tolist() == ref["q"].tolist(), [(hex(int(x[i, j])), hex(int(got[i, j])), hex(int(ref["q"][i, j]))) for i, j in zip(*bad)][:20]
    check_state_tensor(st, ref, fmt, ref["overflow"], ref["underflow"])


@pytest.mark.parametrize("fi,fmt", FMTS)
@pytest.mark.parametrize("k", [-20, -7, -1, 3, 10, 40])
def test_every_bf16_pattern_power_of_two_scales(g, fi, fmt, k):
    """Scale 2^k through a one-entry history (delayed mode): amax_eff = FP8_MAX / 2^k."""
    x = all_bf16_patterns()
    xd = dev_bf16(x)
    st = g.TensorState(hist_len=4)
    mx = fp8.fp8_max(fmt)
    a = np.float32(mx * 2.0 ** (-k))
    st.amax_history[0] = float(a)
    st.hist_count[0] = 1
    q = empty_u8(512, 128)
    g.fp8_quantize(xd, 512, 128, 128, fi, g.FP8_GRAN_TENSOR, g.FP8_SCALE_DELAYED, st, q)
    s, d = quant.scales_from_amax(a, fmt)
    ref_q, ov, un = quant.cast_with_scale(x, s, fmt)
    assert np.array_equal(host_u8(q), ref_q)
    snap = st.snapshot()
    assert np.float32(snap["scale"]) == s and np.float32(snap["scale_inv"]) == d
    assert snap["overflow"] == ov and snap["underflow"] == un
    assert np.float32(snap["amax_cur"]) == quant.amax(x)


@pytest.mark.parametrize("fi,fmt", FMTS)
def test_every_bf16_pattern_random_scales(g, fi, fmt):
    rng = np.random.default_rng(5)
    x = all_bf16_patterns()
    xd = dev_bf16(x)
    for a in rng.uniform(1e-3, 1e3, size=6).astype(np.float32):
        st = g.TensorState(hist_len=2)
        st.amax_history[0] = float(a)
        st.hist_count[0] = 1
        q = empty_u8(512, 128)
        g.fp8_quantize(xd, 512, 128, 128, fi, g.FP8_GRAN_TENSOR, g.FP8_SCALE_DELAYED, st, q)
        s, _ = quant.scales_from_amax(a, fmt)
        ref_q, ov, un = quant.cast_with_scale(x, s, fmt)
        assert np.array_equal(host_u8(q), ref_q)
        snap = st.snapshot()
        assert snap["overflow"] == ov and snap["underflow"] == un


SHAPES_FLAT = [(1, 1), (3, 5), (7, 33), (257, 129), (1000, 1000), (64, 768)]


@pytest.mark.parametrize("fi,fmt", FMTS)
@pytest.mark.parametrize("shape", SHAPES_FLAT)
def test_per_tensor_current_flat(g, fi, fmt, shape):
    R, C = shape
    x = normal_bf16(R * 7 + C, shape, std=3.0) if fi == 0 else lognormal_grad_bf16(R + C, shape)
    st = g.TensorState()
    q = empty_u8(R, C)
    g.fp8_quantize(dev_bf16(x), R, C, C, fi, g.FP8_GRAN_TENSOR, g.FP8_SCALE_CURRENT, st, q)
    ref = quant.quantize_tensor(x, fmt)
    assert np.array_equal(host_u8(q), ref["q"])
    check_state_tensor(st, ref, fmt, ref["overflow"], ref["underflow"])


def test_per_tensor_strided_input(g):
    R, C, ld = 37, 100, 136
    full = normal_bf16(9, (R, ld))
    x = full[:, :C].copy()
    st = g.TensorState()
    q = empty_u8(R, C)
    g.fp8_quantize(dev_bf16(full), R, C, ld, 0, g.FP8_GRAN_TENSOR, g.FP8_SCALE_CURRENT, st, q)
    ref = quant.quantize_tensor(x, fp8.E4M3)
    assert np.array_equal(host_u8(q), ref["q"])
    check_state_tensor(st, ref, fp8.E4M3, ref["overflow"], ref["underflow"])


SHAPES_TILE = [(16, 8), (144, 200), (256, 384), (1040, 776), (128, 128)]


@pytest.mark.parametrize("fi,fmt", FMTS)
@pytest.mark.parametrize("shape", SHAPES_TILE)
@pytest.mark.parametrize("mode", [0, 1])
def test_per_tensor_with_transpose(g, fi, fmt, shape, mode):
    R, C = shape
    x = outlier_normal_bf16(R + 3 * C, shape)
    st = g.TensorState()
    if mode == 1:  # delayed with a history that saturates the outliers
        st.amax_history[:3] = torch.tensor([2.0, 3.5, 1.0])
        st.hist_count[0] = 3
    q = empty_u8(R, C)
    qT = empty_u8(C, R)
    g.fp8_quantize(dev_bf16(x), R, C, C, fi, g.FP8_GRAN_TENSOR, mode, st, q, qT)
    if mode == 0:
        ref = quant.quantize_tensor(x, fmt)
        s = ref["s"]
    else:
        s, _ = quant.scales_from_amax(np.float32(3.5), fmt)
    ref_q, ov, un = quant.cast_with_scale(x, s, fmt)
    assert np.array_equal(host_u8(q), ref_q)
    assert np.array_equal(host_u8(qT), ref_q.T)
    snap = st.snapshot()
    assert snap["overflow"] == ov and snap["underflow"] == un
    assert np.float32(snap["scale"]) == s
    assert np.float32(snap["amax_cur"]) == quant.amax(x)


def test_transpose_only_output(g):
    R, C = 256, 512
    x = normal_bf16(77, (R, C), 0.02)
    st = g.TensorState()
    qT = empty_u8(C, R)
    g.fp8_quantize(dev_bf16(x), R, C, C, 0, g.FP8_GRAN_TENSOR, 0, st, None, qT)
    ref = quant.quantize_tensor(x, fp8.E4M3)
    assert np.array_equal(host_u8(qT), ref["qT"])


@pytest.mark.parametrize("fi,fmt", FMTS)
@pytest.mark.parametrize("shape", [(1, 128), (37, 256), (1000, 1024), (16, 4096)])
def test_tile_1x128(g, fi, fmt, shape):
    R, C = shape
    x = channel_scaled_bf16(R + C, shape)
    q = empty_u8(R, C)
    si = torch.empty(R, C // 128, dtype=torch.float32, device="cuda")
    st = g.TensorState()
    g.fp8_quantize(dev_bf16(x), R, C, C, fi, g.FP8_GRAN_TILE_1x128, 0, st, q, None, si)
    ref = quant.quantize_tile_1x128(x, fmt)
    assert np.array_equal(host_u8(q), ref["q"])
    assert np.array_equal(si.cpu().numpy(), ref["d"])
    snap = st.snapshot()
    assert snap["overflow"] == ref["overflow"] and snap["underflow"] == ref["underflow"]
    assert np.float32(snap["amax_cur"]) == quant.amax(x)


@pytest.mark.parametrize("fi,fmt", FMTS)
@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (512, 1024)])
def test_block_128x128(g, fi, fmt, shape):
    R, C = shape
    x = channel_scaled_bf16(R * 3 + C, shape)
    q = empty_u8(R, C)
    qT = empty_u8(C, R)
    si = torch.empty(R // 128, C // 128, dtype=torch.float32, device="cuda")
    st = g.TensorState()
    g.fp8_quantize(dev_bf16(x), R, C, C, fi, g.FP8_GRAN_BLOCK_128x128, 0, st, q, qT, si)
    ref = quant.quantize_block_128x128(x, fmt)
    assert np.array_equal(host_u8(q), ref["q"])
    assert np.array_equal(host_u8(qT), ref["qT"])
    assert np.array_equal(si.cpu().numpy(), ref["d"])
    snap = st.snapshot()
    assert snap["overflow"] == ref["overflow"] and snap["underflow"] == ref["underflow"]


def test_special_values_inside_tensors(g):
    vals = np.array([np.nan, -np.nan, np.inf, -np.inf, -0.0, 0.0, 1e-30, -1e-30, 3.0, -7.5] * 13, dtype=np.float32)
    x = bf16_bits_from_f32(vals).reshape(10, 13)
    for fi, fmt in FMTS:
        st = g.TensorState()
        q = empty_u8(10, 13)
        g.fp8_quantize(dev_bf16(x), 10, 13, 13, fi, g.FP8_GRAN_TENSOR, 0, st, q)
        ref = quant.quantize_tensor(x, fmt)
        assert np.array_equal(host_u8(q), ref["q"])
        check_state_tensor(st, ref, fmt, ref["overflow"], ref["underflow"])
    # NaN-free with a finite amax: the scale is applied
    x2 = bf16_bits_from_f32(np.array([[np.nan, 1.0, -0.0, -2.0] * 4] * 16, dtype=np.float32))
    st = g.TensorState()
    q = empty_u8(16, 16)
    qT = empty_u8(16, 16)
    g.fp8_quantize(dev_bf16(x2), 16, 16, 16, 0, g.FP8_GRAN_TENSOR, 0, st, q, qT)
    ref = quant.quantize_tensor(x2, fp8.E4M3)
    assert ref["s"] == 224.0
    assert np.array_equal(host_u8(q), ref["q"]) and np.array_equal(host_u8(qT), ref["qT"])


def test_delayed_bootstrap_and_commit(g):
    st = g.TensorState(hist_len=3)
    ost = quant.DelayedState(hist_len=3)
    for t, scale in enumerate([1.0, 0.5, 4.0, 0.25, 8.0, 1.0]):
        x = bf16_bits_from_f32(quant.widen_bf16(normal_bf16(40 + t, (64, 96))) * np.float32(scale))
        q = empty_u8(64, 96)
        g.fp8_quantize(dev_bf16(x), 64, 96, 96, 1, g.FP8_GRAN_TENSOR, g.FP8_SCALE_DELAYED, st, q)
        ref = ost.quantize(x, fp8.E5M2, delayed=True)
        assert np.array_equal(host_u8(q), ref["q"]), t
        g.fp8_history_commit(st)
        ost.commit()
        snap = st.snapshot()
        o = ost.snapshot()
        assert snap["count"] == o["count"]
        assert np.array_equal(snap["hist"], o["hist"])
        assert np.float32(snap["scale"]) == o["scale"] and np.float32(snap["amax_cur"]) == o["amax_cur"]
        assert snap["overflow"] == o["overflow"] and snap["underflow"] == o["underflow"]


@pytest.mark.parametrize("tiled", [False, True])
def test_delayed_running_max_and_commit_reset(g, tiled):
    """amax_cur is the running maximum of the delayed casts since the last commit, the bootstrap
    scale included (the bootstrap amax kernel, then the cast as a plain launch), and the commit
    resets it; a current-scaling cast sets it to its own amax. Against the oracle's state."""
    st, ost = g.TensorState(hist_len=2), quant.DelayedState(hist_len=2)
    R, C = 64, 128
    for t, (scale, mode) in enumerate([(3.0, 1), (0.5, 1), (6.0, 1), (None, "commit"), (0.25, 1), (2.0, 1),
                                        (0.125, 0), (None, "commit"), (9.0, 1)]):
        if mode == "commit":
            g.fp8_history_commit(st)
            ost.commit()
        else:
            x = bf16_bits_from_f32(quant.widen_bf16(normal_bf16(600 + t, (R, C))) * np.float32(scale))
            q, qT = empty_u8(R, C), (empty_u8(C, R) if tiled else None)
            g.fp8_quantize(dev_bf16(x), R, C, C, 1, g.FP8_GRAN_TENSOR, mode, st, q, qT)
            ref = ost.quantize(x, fp8.E5M2, delayed=(mode == 1))
            assert np.array_equal(host_u8(q), ref["q"]), t
            if tiled:
                assert np.array_equal(host_u8(qT), ref["qT"]), t
        snap, o = st.snapshot(), ost.snapshot()
        assert np.float32(snap["amax_cur"]) == o["amax_cur"], t
        assert np.float32(snap["scale"]) == o["scale"] and snap["count"] == o["count"], t
        assert np.array_equal(snap["hist"], o["hist"]), t
        assert snap["overflow"] == o["overflow"] and snap["underflow"] == o["underflow"], t


def test_empty_tensor_writes_unit_scales(g):
    st = g.TensorState()
    st.scale.fill_(5.0)
    q = empty_u8(1)
    g.fp8_quantize(dev_bf16(np.zeros((1,), dtype=np.uint16)), 0, 0, 0, 0, g.FP8_GRAN_TENSOR, 0, st, q)
    snap = st.snapshot()
    assert snap["scale"] == 1.0 and snap["scale_inv"] == 1.0 and snap["amax_cur"] == 0.0


def test_rejections(g):
    st = g.TensorState()
    x = dev_bf16(normal_bf16(1, (16, 16)))
    q = empty_u8(16, 16)
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_quantize(x, 16, 16, 16, 0, g.FP8_GRAN_TILE_1x128, 0, st, q, None, None)
    assert e.value.status in (g.FP8_ERR_INVALID_ARG, g.FP8_ERR_UNSUPPORTED)
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_quantize(x, 16, 16, 16, 7, g.FP8_GRAN_TENSOR, 0, st, q)
    assert e.value.status == g.FP8_ERR_INVALID_ARG
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_quantize(x.data_ptr() + 2, 15, 16, 16, 0, g.FP8_GRAN_TENSOR, 0, st, q)
    assert e.value.status == g.FP8_ERR_ALIGNMENT
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_quantize(x, 16, 16, 16, 0, g.FP8_GRAN_TENSOR, 0, None, q)
    assert e.value.status == g.FP8_ERR_INVALID_ARG


def test_bounded_wait_reports_timeout(g):
    """A wait on a barrier nothing completes runs out after ~50 ms and reports a status;
    the context stays usable afterwards."""
    assert g.fp8_selftest_wait_timeout(50_000_000) == g.FP8_ERR_TIMEOUT
    g.fp8_poll_device_error()  # cleared
    x = dev_bf16(normal_bf16(2, (8, 8)))
    st = g.TensorState()
    q = empty_u8(8, 8)
    g.fp8_quantize(x, 8, 8, 8, 0, g.FP8_GRAN_TENSOR, 0, st, q)
    torch.cuda.synchronize()


def test_subnormal_amax_keeps_unit_scales(g):
    """amax = the smallest bf16 subnormal: FP8_MAX / amax overflows float32, so the pair is
    1, 1 (zeros stay zero codes instead of 0 * inf = NaN); codes and counters as the oracle."""
    x = np.array([[0x0001, 0x0000, 0x8001, 0x8000] * 4] * 16, dtype=np.uint16)
    for fi, fmt in FMTS:
        for qT in (False, True):
            st = g.TensorState()
            q = empty_u8(16, 16)
            t = empty_u8(16, 16) if qT else None
            g.fp8_quantize(dev_bf16(x), 16, 16, 16, fi, g.FP8_GRAN_TENSOR, 0, st, q, t)
            ref = quant.quantize_tensor(x, fmt)
            assert ref["s"] == 1.0 and ref["d"] == 1.0
            assert np.array_equal(host_u8(q), ref["q"])
            check_state_tensor(st, ref, fmt, ref["overflow"], ref["underflow"])


def test_commit_many_matches_single_commits(g):
    """One launch pushing three states equals three single pushes; duplicates are refused."""
    xs = [normal_bf16(60 + i, (32, 64), std=2.0 ** i) for i in range(3)]
    a = [g.TensorState(hist_len=4) for _ in range(3)]
    b = [g.TensorState(hist_len=4) for _ in range(3)]
    for step in range(6):
        for i in range(3):
            for st in (a[i], b[i]):
                q = empty_u8(32, 64)
                g.fp8_quantize(dev_bf16(xs[i]), 32, 64, 64, 0, g.FP8_GRAN_TENSOR, g.FP8_SCALE_DELAYED, st, q)
        g.fp8_history_commit_many(a)
        for st in b:
            g.fp8_history_commit(st)
    for sa, sb in zip(a, b):
        x, y = sa.snapshot(), sb.snapshot()
        assert x["count"] == y["count"] == 6 and np.array_equal(x["hist"], y["hist"])
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_history_commit_many([a[0], a[1], a[0]])
    assert e.value.status == g.FP8_ERR_INVALID_ARG
