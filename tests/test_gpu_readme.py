"""The README's usage example runs as written, and its forward output is the scaled product
of the FP8 codes it made (the oracle's GEMM on sampled outputs, within the GEMM bound)."""
import os
import re

import numpy as np
import pytest
import torch

from oracle import fp8, gemm

from gpu_util import host_bf16_f64, host_u8

pytestmark = pytest.mark.gpu

README = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "README.md")


def test_readme_example_runs_and_matches_the_oracle():
    block = re.search(r"```python\n(.*?)```", open(README).read(), re.S).group(1)
    env = {}
    torch.manual_seed(0)
    exec(compile(block, "README.md", "exec"), env)
    torch.cuda.synchronize()
    env["g"].fp8_poll_device_error()
    M, N = env["M"], env["N"]
    xq, wqT, y = host_u8(env["xq"]), host_u8(env["wqT"]), host_bf16_f64(env["y"])
    d_x, d_w = np.float32(env["xs"].scale_inv.item()), np.float32(env["ws"].scale_inv.item())
    rng = np.random.default_rng(0)
    r, c = rng.integers(0, M, 4096), rng.integers(0, N, 4096)
    ref, mag = gemm.scaled_mm_sampled(xq, fp8.E4M3, wqT, fp8.E4M3, d_x, d_w, r, c)
    assert gemm.within_bound(y[r, c], ref, mag).all()
    assert np.abs(y).max() > 0
