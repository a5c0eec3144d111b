"""Forward / backward of the FP8 up-projection and the delayed-scaling training loop
(oracle; test infrastructure).

Sources:
* "#84 FP8 Precision" page, "Hardware precision": the MLP up-projection (d_model ->
  4 d_model) runs in FP8; the bf16 master weights live in the optimizer and the FP8
  compute copy is re-quantised after each optimizer step and cached for the next
  forward.  "Explanation": the transposed layout gives the matmul both operands
  contiguous along the contraction dimension.
* "FP8 stability guardrails" page, "What an interviewer would ask next": E4M3 for the
  forward operands, E5M2 for the backward signal; "Real products, models, and
  research": delayed scaling with an amax history.

Layouts: x [M,K], W [K,N] (row-major bf16), y = x W [M,N], dy [M,N].
    forward: y  = mm(xq [M,K],  WqT [N,K])          d_x * d_w
    dgrad:   dx = mm(dyq [M,N], Wq [K,N])           d_dy * d_w   (contraction over N)
    wgrad:   dW = mm(xqT [K,M], dyqT [N,M])         d_x * d_dy   (contraction over M)
where mm(A, B) contracts the last axis of both.

Training loop (one step, for each layer): perturb the master weight
W <- bf16(float(W) + delta) (from step 1 on), re-quantise W, cast x and run the
forward, cast dy and run dgrad and wgrad, then push the x, W and dy amaxes into
their histories.  The weight cast uses the weight history before its own push.
"""
from __future__ import annotations

import numpy as np

from . import fp8, gemm, quant


def forward(x_bits, wq_t, d_w, x_state: quant.DelayedState, delayed: bool):
    xo = x_state.quantize(x_bits, fp8.E4M3, delayed=delayed)
    y, mag, _ = gemm.scaled_mm(xo["q"], fp8.E4M3, wq_t, fp8.E4M3, xo["d"], d_w)
    return xo, y, mag


def backward(dy_bits, xo, wq, d_w, dy_state: quant.DelayedState, delayed: bool):
    go = dy_state.quantize(dy_bits, fp8.E5M2, delayed=delayed)
    dx, mag_dx, _ = gemm.scaled_mm(go["q"], fp8.E5M2, wq, fp8.E4M3, go["d"], d_w)
    dw, mag_dw, _ = gemm.scaled_mm(xo["qT"], fp8.E4M3, go["qT"], fp8.E5M2, xo["d"], go["d"])
    return go, dx, mag_dx, dw, mag_dw


def perturb_master(w_bits, delta_f32):
    """Simulated optimizer step: W <- bf16_rne(float32(W) + delta), one fp32 add."""
    w = quant.widen_bf16(w_bits)
    s = (w + np.asarray(delta_f32, dtype=np.float32)).astype(np.float32)
    return _bf16_bits_rne(s)


def _bf16_bits_rne(a):
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    return ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def training_loop(x_bits, dy_bits, w_bits_list, steps, hist_len, delta_fn, with_gemm=True, on_step=None):
    """Delayed-scaling loop over all layers and steps.  ``delta_fn(layer, step)`` returns
    the float32 perturbation.  ``on_step(step, layer, record)`` sees every layer-step."""
    L = len(w_bits_list)
    wst = [quant.DelayedState(hist_len) for _ in range(L)]
    xst = [quant.DelayedState(hist_len) for _ in range(L)]
    gst = [quant.DelayedState(hist_len) for _ in range(L)]
    w = [np.array(b, copy=True) for b in w_bits_list]
    for t in range(steps):
        for l in range(L):
            if t >= 1:
                w[l] = perturb_master(w[l], delta_fn(l, t))
            wo = wst[l].quantize(w[l], fp8.E4M3, delayed=True)
            xo = xst[l].quantize(x_bits, fp8.E4M3, delayed=True)
            go = gst[l].quantize(dy_bits, fp8.E5M2, delayed=True)
            rec = dict(w=wo, x=xo, dy=go, w_master=w[l])
            if with_gemm:
                rec["y"] = gemm.scaled_mm(xo["q"], fp8.E4M3, wo["qT"], fp8.E4M3, xo["d"], wo["d"])[:2]
                rec["dx"] = gemm.scaled_mm(go["q"], fp8.E5M2, wo["q"], fp8.E4M3, go["d"], wo["d"])[:2]
                rec["dw"] = gemm.scaled_mm(xo["qT"], fp8.E4M3, go["qT"], fp8.E5M2, xo["d"], go["d"])[:2]
            wst[l].commit()
            xst[l].commit()
            gst[l].commit()
            rec["state"] = dict(w=wst[l].snapshot(), x=xst[l].snapshot(), dy=gst[l].snapshot())
            if on_step is not None:
                on_step(t, l, rec)
    return wst, xst, gst, w
