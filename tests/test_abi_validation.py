"""The C ABI's synchronous argument checks, on CPU: every call below is refused before it
touches the GPU, with the status include/fp8gb.h documents and a message naming the call.
Device addresses here are made-up numbers (16-byte aligned or deliberately not); each case
fails a host-side check, so nothing is ever dereferenced. The module does not run where a
GPU is present."""
import pytest

torch = pytest.importorskip("torch")
if torch.cuda.is_available():
    pytest.skip("host-side checks only: made-up device addresses", allow_module_level=True)

A16, B16, C16, S16 = 0x10000, 0x20000, 0x30000, 0x40000  # aligned placeholders
ODD = 0x10001                                               # misaligned


@pytest.fixture(scope="module")
def g():
    import __graft_entry__
    try:
        __graft_entry__._build_module().build()
    except RuntimeError as e:
        pytest.skip(f"no CUDA toolkit to build with: {e}")
    import fp8_mixed_precision_saturating_gb300 as m
    return m


def state(g, hist_len=16, base=0x50000):
    return g.fp8_tensor_state_t(base, base + 0x100, base + 0x200, base + 0x210, base + 0x220, base + 0x240, hist_len)


def refused(g, status, who, fn, *args):
    with pytest.raises(g.Fp8Error) as e:
        fn(*args)
    assert e.value.status == status, (e.value.status, str(e.value))
    assert who in str(e.value)


def test_quantize_checks(g):
    st = state(g)
    q = g.fp8_quantize
    refused(g, g.FP8_ERR_INVALID_ARG, "negative", q, A16, -1, 16, 16, 0, 0, 0, st, B16)
    refused(g, g.FP8_ERR_INVALID_ARG, "unknown format", q, A16, 16, 16, 16, 7, 0, 0, st, B16)
    refused(g, g.FP8_ERR_INVALID_ARG, "granularity", q, A16, 16, 16, 16, 0, 9, 0, st, B16)
    refused(g, g.FP8_ERR_INVALID_ARG, "scaling mode", q, A16, 16, 16, 16, 0, 0, 5, st, B16)
    refused(g, g.FP8_ERR_INVALID_ARG, "ld", q, A16, 16, 16, 8, 0, 0, 0, st, B16)
    refused(g, g.FP8_ERR_INVALID_ARG, "null input", q, None, 16, 16, 16, 0, 0, 0, st, B16)
    refused(g, g.FP8_ERR_INVALID_ARG, "no output", q, A16, 16, 16, 16, 0, 0, 0, st, None)
    refused(g, g.FP8_ERR_ALIGNMENT, "aligned", q, ODD, 16, 16, 16, 0, 0, 0, st, B16)
    refused(g, g.FP8_ERR_ALIGNMENT, "aligned", q, A16, 16, 16, 16, 0, 0, 0, st, ODD)
    # layouts the tiled kernels do not take
    refused(g, g.FP8_ERR_UNSUPPORTED, "multiples of 8", q, A16, 16, 12, 12, 0, 0, 0, st, B16, C16)
    refused(g, g.FP8_ERR_UNSUPPORTED, "rows % 16", q, A16, 8, 16, 16, 0, 0, 0, st, B16, C16)
    refused(g, g.FP8_ERR_UNSUPPORTED, "cols % 128", q, A16, 16, 64, 64, 0, g.FP8_GRAN_TILE_1x128, 0, None, B16,
            None, S16)
    refused(g, g.FP8_ERR_UNSUPPORTED, "current scaling", q, A16, 128, 128, 128, 0, g.FP8_GRAN_BLOCK_128x128,
            g.FP8_SCALE_DELAYED, None, B16, None, S16)
    refused(g, g.FP8_ERR_UNSUPPORTED, "65535", q, A16, 128 * 65536, 128, 128, 0, g.FP8_GRAN_BLOCK_128x128, 0,
            None, B16, None, S16)
    # delayed scaling needs a history
    refused(g, g.FP8_ERR_INVALID_ARG, "history", q, A16, 16, 16, 16, 0, 0, g.FP8_SCALE_DELAYED,
            g.fp8_tensor_state_t(0, 0, S16, S16 + 16, S16 + 32, S16 + 64, 0), B16)


def test_scaled_mm_checks(g):
    mm = g.fp8_scaled_mm
    refused(g, g.FP8_ERR_INVALID_ARG, "negative", mm, A16, 0, B16, 0, -1, 16, 16, 16, 16, 0, S16, S16, C16, 16)
    refused(g, g.FP8_ERR_INVALID_ARG, "format", mm, A16, 3, B16, 0, 16, 16, 16, 16, 16, 0, S16, S16, C16, 16)
    refused(g, g.FP8_ERR_INVALID_ARG, "granularity", mm, A16, 0, B16, 0, 16, 16, 16, 16, 16,
            g.FP8_GRAN_TILE_1x128, S16, S16, C16, 16)
    refused(g, g.FP8_ERR_INVALID_ARG, "null C", mm, A16, 0, B16, 0, 16, 16, 16, 16, 16, 0, S16, S16, None, 16)
    refused(g, g.FP8_ERR_INVALID_ARG, "ldc", mm, A16, 0, B16, 0, 16, 32, 16, 16, 16, 0, S16, S16, C16, 16)
    refused(g, g.FP8_ERR_ALIGNMENT, "aligned", mm, A16, 0, B16, 0, 16, 16, 16, 16, 16, 0, S16, S16, ODD, 16)
    refused(g, g.FP8_ERR_INVALID_ARG, "null A", mm, None, 0, B16, 0, 16, 16, 16, 16, 16, 0, S16, S16, C16, 16)
    refused(g, g.FP8_ERR_INVALID_ARG, "lda", mm, A16, 0, B16, 0, 16, 16, 32, 16, 32, 0, S16, S16, C16, 16)
    refused(g, g.FP8_ERR_ALIGNMENT, "aligned", mm, A16, 0, B16, 0, 16, 16, 16, 24, 16, 0, S16, S16, C16, 16)
    refused(g, g.FP8_ERR_UNSUPPORTED, "multiples of 128", mm, A16, 0, B16, 0, 128, 128, 64, 64, 64,
            g.FP8_GRAN_BLOCK_128x128, S16, S16, C16, 128)
    refused(g, g.FP8_ERR_UNSUPPORTED, "2^31", mm, A16, 0, B16, 0, 1 << 31, 16, 16, 16, 16, 0, S16, S16, C16, 16)


def test_grouped_and_many_checks(g):
    p = g.mm_problem(A16, 0, B16, 0, 16, 16, 16, 16, 16, S16, S16, C16, 16)
    refused(g, g.FP8_ERR_INVALID_ARG, "1 or 2 problems", g.fp8_scaled_mm_grouped, [p, p, p])
    refused(g, g.FP8_ERR_INVALID_ARG, "negative workspace", g.fp8_scaled_mm_grouped, [p, p], C16, -1)
    refused(g, g.FP8_ERR_ALIGNMENT, "workspace", g.fp8_scaled_mm_grouped, [p, p], ODD, 64)
    bad_mn = g.mm_problem(A16, 0, B16, 0, 16, 16, 16, 16, 16, S16, S16, C16, 16, mn_major=2)
    refused(g, g.FP8_ERR_INVALID_ARG, "mn_major is 0 or 1", g.fp8_scaled_mm_grouped, [p, bad_mn])
    short_mn = g.mm_problem(A16, 0, B16, 0, 32, 16, 16, 16, 16, S16, S16, C16, 16, mn_major=1)  # lda < M
    refused(g, g.FP8_ERR_INVALID_ARG, "leading dimension", g.fp8_scaled_mm_grouped, [p, short_mn])
    sa, sb = state(g, base=0x50000), state(g, base=0x60000)
    j = g.quant_job(A16, 16, 16, 16, 0, 0, sa, B16, C16)
    refused(g, g.FP8_ERR_INVALID_ARG, "jobs", g.fp8_quantize_many, [])
    refused(g, g.FP8_ERR_INVALID_ARG, "jobs", g.fp8_quantize_many, [j] * 5)
    refused(g, g.FP8_ERR_INVALID_ARG, "repeated", g.fp8_quantize_many, [j, g.quant_job(A16, 16, 16, 16, 0, 0, sa, B16, C16)])
    refused(g, g.FP8_ERR_INVALID_ARG, "scaling mode",
            g.fp8_quantize_many, [j, g.quant_job(A16, 16, 16, 16, 0, 4, sb, B16, C16)])


def test_layer_and_state_checks(g):
    sw, sx, sg = state(g, base=0x50000), state(g, base=0x60000), state(g, base=0x70000)
    refused(g, g.FP8_ERR_INVALID_ARG, "negative", g.fp8_linear_fwd, A16, -16, 16, 16, B16, sw, None, sx, 0, 0,
            C16, None, None, S16)
    refused(g, g.FP8_ERR_INVALID_ARG, "required", g.fp8_linear_fwd, A16, 16, 16, 16, B16, sw, None, sx, 0, 0,
            None, None, None, S16)
    refused(g, g.FP8_ERR_UNSUPPORTED, "multiples of 16", g.fp8_linear_bwd, A16, 24, 16, 16, B16, sx, C16, sw, sg,
            0, S16, S16, A16, B16)
    refused(g, g.FP8_ERR_INVALID_ARG, "dyq_ws", g.fp8_linear_bwd, A16, 16, 16, 16, B16, sx, C16, sw, sg, 0, None,
            S16, A16, B16)
    refused(g, g.FP8_ERR_INVALID_ARG, "mode", g.fp8_update_requantize_weights, A16, B16, 16, 16, 3, sw, C16, S16)
    refused(g, g.FP8_ERR_UNSUPPORTED, "multiples of 8", g.fp8_update_requantize_weights, A16, B16, 16, 12, 0, sw,
            C16, None)
    many = [state(g, base=0x100000 + 0x1000 * i) for i in range(33)]
    refused(g, g.FP8_ERR_INVALID_ARG, "states per call", g.fp8_history_commit_many, many)
    refused(g, g.FP8_ERR_INVALID_ARG, "needs amax_history", g.fp8_history_commit_many,
            [g.fp8_tensor_state_t(0, 0, S16, S16, S16, S16, 16)])
    refused(g, g.FP8_ERR_INVALID_ARG, "twice", g.fp8_history_commit_many, [sw, sx, sw])
