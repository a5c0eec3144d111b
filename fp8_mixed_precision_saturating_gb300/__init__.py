"""Python binding of libfp8gb (the GB300 FP8 up-projection library).

Argument marshalling only: every entry point forwards to the C ABI of the same name
declared in include/fp8gb.h, and every step of the computation runs in the library's
CUDA kernels. Tensors may be passed as torch tensors (their ``data_ptr()`` is used) or as
raw integer device addresses; ``stream`` may be a torch.cuda.Stream, an integer handle
or None (the current torch stream when torch is importable, else the default stream).

There is no fallback: importing this package fails loudly when libfp8gb.so has not been
built (``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8gb.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libfp8gb.so is missing at {LIB_PATH}: build it first (fp8_mixed_precision_saturating_gb300._build.build())")

lib = ctypes.CDLL(LIB_PATH)

# enums (include/fp8gb.h)
FP8_OK, FP8_ERR_INVALID_ARG, FP8_ERR_UNSUPPORTED, FP8_ERR_ALIGNMENT, FP8_ERR_CUDA, FP8_ERR_TIMEOUT = range(6)
FP8_E4M3, FP8_E5M2 = 0, 1
FP8_GRAN_TENSOR, FP8_GRAN_TILE_1x128, FP8_GRAN_BLOCK_128x128, FP8_GRAN_MX_1x32 = 0, 1, 2, 3
FP8_SCALE_CURRENT, FP8_SCALE_DELAYED = 0, 1


class fp8_tensor_state_t(ctypes.Structure):
    _fields_ = [
        ("amax_history", ctypes.c_void_p),
        ("hist_count", ctypes.c_void_p),
        ("scale", ctypes.c_void_p),
        ("scale_inv", ctypes.c_void_p),
        ("amax_cur", ctypes.c_void_p),
        ("counters", ctypes.c_void_p),
        ("hist_len", ctypes.c_int32),
    ]


class fp8_mm_problem_t(ctypes.Structure):
    _fields_ = [
        ("A", ctypes.c_void_p),
        ("fa", ctypes.c_int),
        ("B", ctypes.c_void_p),
        ("fb", ctypes.c_int),
        ("M", ctypes.c_int64),
        ("N", ctypes.c_int64),
        ("K", ctypes.c_int64),
        ("lda", ctypes.c_int64),
        ("ldb", ctypes.c_int64),
        ("scale_inv_a", ctypes.c_void_p),
        ("scale_inv_b", ctypes.c_void_p),
        ("C_bf16", ctypes.c_void_p),
        ("ldc", ctypes.c_int64),
        ("mn_major", ctypes.c_int32),
    ]


class fp8_quant_job_t(ctypes.Structure):
    _fields_ = [
        ("x_bf16", ctypes.c_void_p),
        ("rows", ctypes.c_int64),
        ("cols", ctypes.c_int64),
        ("ld", ctypes.c_int64),
        ("fmt", ctypes.c_int),
        ("mode", ctypes.c_int),
        ("st", ctypes.POINTER(fp8_tensor_state_t)),
        ("q_out", ctypes.c_void_p),
        ("qT_out", ctypes.c_void_p),
    ]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_SP = ctypes.POINTER(fp8_tensor_state_t)
_MP = ctypes.POINTER(fp8_mm_problem_t)

_SIGS = {
    "fp8_quantize": [_P, _I64, _I64, _I64, _I, _I, _I, _SP, _P, _P, _P, _P],
    "fp8_scaled_mm": [_P, _I, _P, _I, _I64, _I64, _I64, _I64, _I64, _I, _P, _P, _P, _I64, _P],
    "fp8_scaled_mm_ws": [_P, _I, _P, _I, _I64, _I64, _I64, _I64, _I64, _I, _P, _P, _P, _I64, _P, _I64, _P],
    "fp8_scaled_mm_grouped": [_MP, ctypes.c_int32, _P, _I64, _P],
    "fp8_quantize_many": [ctypes.POINTER(fp8_quant_job_t), ctypes.c_int32, _P],
    "fp8_scaled_mm_quant": [_P, _I, _P, _I, _I64, _I64, _I64, _I64, _I64, _P, _P, _P, _I64, _I, _SP, _P, _P],
    "fp8_requantize_weights": [_P, _I64, _I64, _I, _I, _SP, _P, _P, _P, _P],
    "fp8_update_requantize_weights": [_P, _P, _I64, _I64, _I, _SP, _P, _P, _P],
    "fp8_linear_fwd": [_P, _I64, _I64, _I64, _P, _SP, _P, _SP, _I, _I, _P, _P, _P, _P, _P],
    "fp8_linear_bwd": [_P, _I64, _I64, _I64, _P, _SP, _P, _SP, _SP, _I, _P, _P, _P, _P, _P],
    "fp8_linear_bwd_noalloc": [_P, _I64, _I64, _I64, _P, _SP, _P, _SP, _SP, _I, _P, _P, _P],
    "fp8_linear_bwd_ws": [_P, _I64, _I64, _I64, _P, _SP, _P, _SP, _SP, _I, _P, _P, _P, _P, _P, _I64, _P],
    "fp8_linear_bwd_mn": [_P, _I64, _I64, _I64, _P, _SP, _P, _SP, _SP, _I, _P, _P, _P, _P, _I64, _P],
    "fp8_scaled_mm_t": [_P, _I, _P, _I, _I64, _I64, _I64, _I64, _I64, _P, _P, _P, _I64, _P, _I64, _P],
    "fp8_history_commit": [_SP, _P],
    "fp8_history_commit_many": [_SP, ctypes.c_int32, _P],
    "fp8_poll_device_error": [],
    "fp8_set_wait_limit_ns": [ctypes.c_ulonglong],
    "fp8_selftest_wait_timeout": [ctypes.c_ulonglong, _P],
    "fp8_get_last_error_detail": [ctypes.c_char_p, ctypes.c_size_t],
}
for _name, _args in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
lib.fp8_scaled_mm_grouped_workspace_bytes.argtypes = [_MP, ctypes.c_int32]
lib.fp8_scaled_mm_grouped_workspace_bytes.restype = ctypes.c_int64
lib.fp8_linear_bwd_workspace_bytes.argtypes = [_I64, _I64, _I64]
lib.fp8_linear_bwd_workspace_bytes.restype = ctypes.c_int64
lib.fp8_scaled_mm_workspace_bytes.argtypes = [_I64, _I64, _I64]
lib.fp8_scaled_mm_workspace_bytes.restype = ctypes.c_int64
lib.fp8_status_string.argtypes = [ctypes.c_int]
lib.fp8_status_string.restype = ctypes.c_char_p


class Fp8Error(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{fp8_status_string(status)}: {detail}")
        self.status = status
        self.detail = detail


def fp8_status_string(s: int) -> str:
    return lib.fp8_status_string(s).decode()


def fp8_get_last_error_detail() -> str:
    buf = ctypes.create_string_buffer(512)
    lib.fp8_get_last_error_detail(buf, 512)
    return buf.value.decode()


def _check(status: int) -> int:
    if status != FP8_OK:
        raise Fp8Error(status, fp8_get_last_error_detail())
    return status


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _state(st):
    if st is None:
        return None
    if isinstance(st, fp8_tensor_state_t):
        return ctypes.byref(st)
    return ctypes.byref(st.c)


class TensorState:
    """Device buffers of one tensor role's scaling state, allocated with torch (plumbing).

    Fields mirror fp8_tensor_state_t: amax_history [hist_len] fp32, hist_count int32,
    scale, scale_inv, amax_cur fp32, counters [2] int64 (read as uint64)."""

    def __init__(self, hist_len: int = 16, device="cuda"):
        import torch
        self.hist_len = hist_len
        self.buf_f = torch.zeros(hist_len + 3, dtype=torch.float32, device=device)
        self.buf_i = torch.zeros(1, dtype=torch.int32, device=device)
        self.buf_c = torch.zeros(2, dtype=torch.int64, device=device)
        self.amax_history = self.buf_f[:hist_len]
        self.scale = self.buf_f[hist_len:hist_len + 1]
        self.scale_inv = self.buf_f[hist_len + 1:hist_len + 2]
        self.amax_cur = self.buf_f[hist_len + 2:hist_len + 3]
        self.hist_count = self.buf_i
        self.counters = self.buf_c
        self.c = fp8_tensor_state_t(
            self.amax_history.data_ptr(), self.hist_count.data_ptr(), self.scale.data_ptr(),
            self.scale_inv.data_ptr(), self.amax_cur.data_ptr(), self.counters.data_ptr(), hist_len)

    def reset(self):
        self.buf_f.zero_()
        self.buf_i.zero_()
        self.buf_c.zero_()

    def snapshot(self) -> dict:
        """Host copy of the state (synchronises)."""
        f = self.buf_f.cpu().numpy()
        h = self.hist_len
        return dict(hist=f[:h].copy(), scale=f[h], scale_inv=f[h + 1], amax_cur=f[h + 2],
                    count=int(self.buf_i.cpu()[0]), overflow=int(self.buf_c.cpu()[0]), underflow=int(self.buf_c.cpu()[1]))


# ---------------------------------------------------------------------------------------
# entry points (same names and argument order as the C ABI)
# ---------------------------------------------------------------------------------------
def fp8_quantize(x, rows, cols, ld, fmt, gran, mode, st, q_out, qT_out=None, unit_scale_inv=None, stream=None):
    return _check(lib.fp8_quantize(_ptr(x), rows, cols, ld, fmt, gran, mode, _state(st), _ptr(q_out), _ptr(qT_out),
                                   _ptr(unit_scale_inv), _stream(stream)))


def fp8_scaled_mm(A, fa, B, fb, M, N, K, lda, ldb, gran, scale_inv_a, scale_inv_b, C, ldc, stream=None):
    return _check(lib.fp8_scaled_mm(_ptr(A), fa, _ptr(B), fb, M, N, K, lda, ldb, gran, _ptr(scale_inv_a),
                                    _ptr(scale_inv_b), _ptr(C), ldc, _stream(stream)))


def fp8_scaled_mm_ws(A, fa, B, fb, M, N, K, lda, ldb, gran, scale_inv_a, scale_inv_b, C, ldc, workspace,
                     workspace_bytes, stream=None):
    return _check(lib.fp8_scaled_mm_ws(_ptr(A), fa, _ptr(B), fb, M, N, K, lda, ldb, gran, _ptr(scale_inv_a),
                                       _ptr(scale_inv_b), _ptr(C), ldc, _ptr(workspace), workspace_bytes,
                                       _stream(stream)))


def quant_job(x, rows, cols, ld, fmt, mode, st, q, qT):
    """One fp8_quant_job_t (per-tensor scale) for fp8_quantize_many; keeps st alive."""
    c = st if isinstance(st, fp8_tensor_state_t) else st.c
    j = fp8_quant_job_t(_ptr(x), rows, cols, ld, fmt, mode, ctypes.pointer(c), _ptr(q), _ptr(qT))
    j._keep = st
    return j


def fp8_quantize_many(jobs, stream=None):
    arr = (fp8_quant_job_t * len(jobs))(*jobs)
    return _check(lib.fp8_quantize_many(arr, len(jobs), _stream(stream)))


def mm_problem(A, fa, B, fb, M, N, K, lda, ldb, scale_inv_a, scale_inv_b, C, ldc, mn_major=0):
    """One fp8_mm_problem_t (per-tensor scales) for fp8_scaled_mm_grouped."""
    return fp8_mm_problem_t(_ptr(A), fa, _ptr(B), fb, M, N, K, lda, ldb, _ptr(scale_inv_a), _ptr(scale_inv_b),
                            _ptr(C), ldc, mn_major)


def fp8_scaled_mm_grouped(problems, workspace=None, workspace_bytes=0, stream=None):
    arr = (fp8_mm_problem_t * len(problems))(*problems)
    return _check(lib.fp8_scaled_mm_grouped(arr, len(problems), _ptr(workspace), workspace_bytes, _stream(stream)))


def fp8_scaled_mm_grouped_workspace_bytes(problems) -> int:
    arr = (fp8_mm_problem_t * len(problems))(*problems)
    n = lib.fp8_scaled_mm_grouped_workspace_bytes(arr, len(problems))
    if n < 0:
        raise Fp8Error(FP8_ERR_INVALID_ARG, fp8_get_last_error_detail())
    return n


def fp8_scaled_mm_workspace_bytes(M, N, K) -> int:
    n = lib.fp8_scaled_mm_workspace_bytes(M, N, K)
    if n < 0:
        raise Fp8Error(FP8_ERR_CUDA, "fp8_scaled_mm_workspace_bytes")
    return n


def fp8_scaled_mm_quant(A, fa, B, fb, M, N, K, lda, ldb, scale_inv_a, scale_inv_b, C, ldc, fc, c_st, Cq,
                        stream=None):
    return _check(lib.fp8_scaled_mm_quant(_ptr(A), fa, _ptr(B), fb, M, N, K, lda, ldb, _ptr(scale_inv_a),
                                          _ptr(scale_inv_b), _ptr(C), ldc, fc, _state(c_st), _ptr(Cq), _stream(stream)))


def fp8_requantize_weights(w_master, K, N, gran, mode, st, wq_kn, wqT_nk, block_scale_inv=None, stream=None):
    return _check(lib.fp8_requantize_weights(_ptr(w_master), K, N, gran, mode, _state(st), _ptr(wq_kn), _ptr(wqT_nk),
                                             _ptr(block_scale_inv), _stream(stream)))


def fp8_update_requantize_weights(w_master, delta, K, N, mode, st, wq_kn, wqT_nk, stream=None):
    return _check(lib.fp8_update_requantize_weights(_ptr(w_master), _ptr(delta), K, N, mode, _state(st), _ptr(wq_kn),
                                                    _ptr(wqT_nk), _stream(stream)))


def fp8_linear_fwd(x, M, K, N, wqT_nk, w_st, w_block_scale_inv, x_st, gran, mode, xq_save, xqT_save,
                   x_tile_scale_inv, y, stream=None):
    return _check(lib.fp8_linear_fwd(_ptr(x), M, K, N, _ptr(wqT_nk), _state(w_st), _ptr(w_block_scale_inv),
                                     _state(x_st), gran, mode, _ptr(xq_save), _ptr(xqT_save), _ptr(x_tile_scale_inv),
                                     _ptr(y), _stream(stream)))


def fp8_linear_bwd(dy, M, K, N, xqT_save, x_st, wq_kn, w_st, dy_st, mode, dyq_ws, dyqT_ws, dx, dw, stream=None):
    return _check(lib.fp8_linear_bwd(_ptr(dy), M, K, N, _ptr(xqT_save), _state(x_st), _ptr(wq_kn), _state(w_st),
                                     _state(dy_st), mode, _ptr(dyq_ws), _ptr(dyqT_ws), _ptr(dx), _ptr(dw),
                                     _stream(stream)))


def fp8_linear_bwd_ws(dy, M, K, N, xqT_save, x_st, wq_kn, w_st, dy_st, mode, dyq_ws, dyqT_ws, dx, dw, workspace,
                      workspace_bytes, stream=None):
    return _check(lib.fp8_linear_bwd_ws(_ptr(dy), M, K, N, _ptr(xqT_save), _state(x_st), _ptr(wq_kn), _state(w_st),
                                        _state(dy_st), mode, _ptr(dyq_ws), _ptr(dyqT_ws), _ptr(dx), _ptr(dw),
                                        _ptr(workspace), workspace_bytes, _stream(stream)))


def fp8_linear_bwd_mn(dy, M, K, N, xq_save, x_st, wq_kn, w_st, dy_st, mode, dyq_ws, dx, dw, workspace=None,
                      workspace_bytes=0, stream=None):
    return _check(lib.fp8_linear_bwd_mn(_ptr(dy), M, K, N, _ptr(xq_save), _state(x_st), _ptr(wq_kn), _state(w_st),
                                        _state(dy_st), mode, _ptr(dyq_ws), _ptr(dx), _ptr(dw), _ptr(workspace),
                                        workspace_bytes, _stream(stream)))


def fp8_scaled_mm_t(A, fa, B, fb, M, N, K, lda, ldb, scale_inv_a, scale_inv_b, C, ldc, workspace=None,
                    workspace_bytes=0, stream=None):
    return _check(lib.fp8_scaled_mm_t(_ptr(A), fa, _ptr(B), fb, M, N, K, lda, ldb, _ptr(scale_inv_a),
                                      _ptr(scale_inv_b), _ptr(C), ldc, _ptr(workspace), workspace_bytes,
                                      _stream(stream)))


def fp8_linear_bwd_workspace_bytes(M, K, N) -> int:
    n = lib.fp8_linear_bwd_workspace_bytes(M, K, N)
    if n < 0:
        raise Fp8Error(FP8_ERR_CUDA, "fp8_linear_bwd_workspace_bytes")
    return n


def fp8_linear_bwd_noalloc(dy, M, K, N, xqT_save, x_st, wq_kn, w_st, dy_st, mode, dx, dw, stream=None):
    """fp8_linear_bwd with the dy codes in the library's static device array (no scratch
    arguments, no allocation by the call); see include/fp8gb.h for the size limit."""
    return _check(lib.fp8_linear_bwd_noalloc(_ptr(dy), M, K, N, _ptr(xqT_save), _state(x_st), _ptr(wq_kn),
                                             _state(w_st), _state(dy_st), mode, _ptr(dx), _ptr(dw), _stream(stream)))


def fp8_history_commit(st, stream=None):
    return _check(lib.fp8_history_commit(_state(st), _stream(stream)))


def fp8_history_commit_many(states, stream=None):
    """Push the amaxes of several distinct states in one launch (at most 32)."""
    arr = (fp8_tensor_state_t * len(states))(*[st if isinstance(st, fp8_tensor_state_t) else st.c for st in states])
    return _check(lib.fp8_history_commit_many(arr, len(states), _stream(stream)))


def fp8_poll_device_error():
    return _check(lib.fp8_poll_device_error())


def fp8_set_wait_limit_ns(ns: int):
    return _check(lib.fp8_set_wait_limit_ns(ns))


def fp8_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    """Returns the raw status (FP8_ERR_TIMEOUT is the expected result)."""
    return lib.fp8_selftest_wait_timeout(limit_ns, _stream(stream))
