"""GPU parity of fp8_quantize_many (several per-tensor quantises in one cooperative launch)
against the CPU oracle: every job's codes, transposed codes, amax, scales, counters and
history bit-exact, as if each had been quantised alone."""
import numpy as np
import pytest
import torch

from datagen import bf16_bits_from_f32, normal_bf16, outlier_normal_bf16
from oracle import fp8, quant

from gpu_util import dev_bf16, empty_u8, host_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import fp8_mixed_precision_saturating_gb300 as m
    return m


def make_job(g, x, fi, mode, st):
    r, c = x.shape
    xd = dev_bf16(x)
    q, qT = empty_u8(r, c), empty_u8(c, r)
    return g.quant_job(xd, r, c, c, fi, mode, st, q, qT), (xd, q, qT)


def check(st, ref, q, qT, o):
    assert np.array_equal(host_u8(q), ref["q"]) and np.array_equal(host_u8(qT), ref["qT"])
    s = st.snapshot()
    assert np.float32(s["amax_cur"]) == o["amax_cur"] and np.float32(s["scale"]) == o["scale"]
    assert np.float32(s["scale_inv"]) == o["scale_inv"]
    assert s["overflow"] == o["overflow"] and s["underflow"] == o["underflow"]
    assert s["count"] == o["count"] and np.array_equal(s["hist"], o["hist"])


@pytest.mark.parametrize("fi,fmt", [(0, fp8.E4M3), (1, fp8.E5M2)])
def test_many_current_scaling(g, fi, fmt):
    # a weight-like and an activation-like tensor, ragged against the 128 x 128 tiles, plus
    # a tensor with outliers that saturate
    xs = [normal_bf16(1, (256, 520), 0.02), normal_bf16(2, (400, 264)), outlier_normal_bf16(3, (1040, 136))]
    sts = [g.TensorState() for _ in xs]
    osts = [quant.DelayedState() for _ in xs]
    jobs, keep = zip(*[make_job(g, x, fi, g.FP8_SCALE_CURRENT, st) for x, st in zip(xs, sts)])
    g.fp8_quantize_many(list(jobs))
    torch.cuda.synchronize()
    for x, st, ost, (_, q, qT) in zip(xs, sts, osts, keep):
        ref = ost.quantize(x, fmt, delayed=False)
        check(st, ref, q, qT, ost.snapshot())
    g.fp8_poll_device_error()


def test_many_delayed_steps_with_commits(g):
    """Bootstrap (own amax) on the first step, delayed scales after it; jobs of one launch
    may be in different phases (a fresh state beside one with history)."""
    hist = 3
    sts = [g.TensorState(hist), g.TensorState(hist)]
    osts = [quant.DelayedState(hist), quant.DelayedState(hist)]
    late = g.TensorState(hist)  # joins at step 2 with an empty history
    olate = quant.DelayedState(hist)
    for t, scale in enumerate([1.0, 0.25, 8.0, 1.0]):
        xs = [bf16_bits_from_f32(quant.widen_bf16(normal_bf16(50 + t, (128, 384), 0.02)) * np.float32(scale)),
              bf16_bits_from_f32(quant.widen_bf16(normal_bf16(60 + t, (512, 256))) * np.float32(scale))]
        all_sts, all_osts = list(sts), list(osts)
        if t >= 2:
            xs.append(normal_bf16(70 + t, (256, 128)))
            all_sts.append(late)
            all_osts.append(olate)
        jobs, keep = zip(*[make_job(g, x, 0, g.FP8_SCALE_DELAYED, st) for x, st in zip(xs, all_sts)])
        g.fp8_quantize_many(list(jobs))
        refs = [o.quantize(x, fp8.E4M3, delayed=True) for x, o in zip(xs, all_osts)]
        g.fp8_history_commit_many(all_sts)
        for o in all_osts:
            o.commit()
        torch.cuda.synchronize()
        for st, ref, o, (_, q, qT) in zip(all_sts, refs, all_osts, keep):
            check(st, ref, q, qT, o.snapshot())
    g.fp8_poll_device_error()


def test_many_history_window_longer_than_a_warp(g):
    """A 40-entry window (the history is read one entry per lane, 32 lanes): before the ring
    wraps only the first `count` entries count; after it wraps all 40 do, and the largest
    entry (step 3's) leaves the window when step 43's amax overwrites it."""
    hist = 40
    sts = [g.TensorState(hist), g.TensorState(hist)]
    osts = [quant.DelayedState(hist), quant.DelayedState(hist)]
    for t in range(46):
        scale = 32.0 if t == 3 else 2.0 ** ((t % 5) - 2)
        xs = [bf16_bits_from_f32(quant.widen_bf16(normal_bf16(200 + t, (64, 256))) * np.float32(scale)),
              bf16_bits_from_f32(quant.widen_bf16(normal_bf16(300 + t, (128, 128), 0.02)) * np.float32(scale))]
        jobs, keep = zip(*[make_job(g, x, 0, g.FP8_SCALE_DELAYED, st) for x, st in zip(xs, sts)])
        g.fp8_quantize_many(list(jobs))
        refs = [o.quantize(x, fp8.E4M3, delayed=True) for x, o in zip(xs, osts)]
        if t in (0, 1, 2, 4, 31, 32, 33, 39, 40, 41, 43, 44, 45):
            torch.cuda.synchronize()
            for st, ref, o, (_, q, qT) in zip(sts, refs, osts, keep):
                check(st, ref, q, qT, o.snapshot())
        g.fp8_history_commit_many(sts)
        for o in osts:
            o.commit()
    g.fp8_poll_device_error()


def test_many_mixed_formats_run_one_by_one(g):
    xs = [normal_bf16(4, (256, 256)), normal_bf16(5, (128, 64))]
    sts = [g.TensorState(), g.TensorState()]
    j0, k0 = make_job(g, xs[0], 0, g.FP8_SCALE_CURRENT, sts[0])
    j1, k1 = make_job(g, xs[1], 1, g.FP8_SCALE_CURRENT, sts[1])
    g.fp8_quantize_many([j0, j1])
    torch.cuda.synchronize()
    for x, fmt, st, (_, q, qT) in ((xs[0], fp8.E4M3, sts[0], k0), (xs[1], fp8.E5M2, sts[1], k1)):
        o = quant.DelayedState()
        ref = o.quantize(x, fmt, delayed=False)
        check(st, ref, q, qT, o.snapshot())


def test_many_rejections(g):
    st = g.TensorState()
    j, keep = make_job(g, normal_bf16(6, (16, 16)), 0, 0, st)
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_quantize_many([j, j])  # one state twice
    assert e.value.status == g.FP8_ERR_INVALID_ARG
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_quantize_many([])
    assert e.value.status == g.FP8_ERR_INVALID_ARG
    others = [make_job(g, normal_bf16(7 + i, (16, 16)), 0, 0, g.TensorState()) for i in range(5)]
    with pytest.raises(g.Fp8Error) as e:
        g.fp8_quantize_many([o[0] for o in others])
    assert e.value.status == g.FP8_ERR_INVALID_ARG
    g.fp8_poll_device_error()
