"""Python binding of libqp (include/qp.h): block-quantized weight dequantization
and the batched-prefill projection on one GB300 (sm_103a).

Argument marshalling only.  Every function has the name of the C entry point
it calls and takes the same arguments; device buffers may be given as torch
tensors (their ``data_ptr()`` is passed) or as raw integer addresses, and
``stream`` as a ``torch.cuda.Stream``, a raw ``cudaStream_t`` integer, or None
for torch's current stream.  A non-OK status raises ``QPError``.  There is no
CPU path: when the CUDA library cannot be built or loaded, ``load()`` raises.
"""
import ctypes
import os

from . import _build

F16, Q8_0, Q2_K, Q4_K, Q5_K, Q6_K = 1, 8, 10, 12, 13, 14
TYPES = {"F16": F16, "Q8_0": Q8_0, "Q2_K": Q2_K, "Q4_K": Q4_K, "Q5_K": Q5_K, "Q6_K": Q6_K}

QP_OK = 0
QP_ERR_INVALID_PARAMETER = 1
QP_ERR_UNSUPPORTED_TYPE = 2
QP_ERR_UNSUPPORTED_SHAPE = 3
QP_ERR_CUDA = 4
QP_ERR_TIMEOUT = 5
QP_ERR_MISALIGNED = 6
QP_ERR_NO_DEVICE = 7
QP_ERR_PAIR_ALLOC = 8

# Every symbol include/qp.h declares.
EXPORTS = ("qp_status_str", "qp_block_info", "qp_row_bytes", "qp_dequant_f32", "qp_dequant_f16",
           "qp_prefill_gemm", "qp_prefill_gemm_f16w", "qp_prefill_gemm_group", "qp_prefill_chunked_group",
           "qp_prefill_chunked", "qp_decode_gemv", "qp_decode_gemv_group", "qp_plan_prefill", "qp_check", "qp_set_wait_limit_ns",
           "qp_debug_inject_stall", "qp_set_gemm_cta_pairs")

QP_MAX_GROUP = 8
QP_GEMV_MAX_T = 8


class QPProjShape(ctypes.Structure):
    """qp_proj_shape: one projection for the fit planner."""
    _fields_ = [("type", ctypes.c_int), ("out_f", ctypes.c_int64), ("in_f", ctypes.c_int64)]


class QPPrefillPlan(ctypes.Structure):
    """qp_prefill_plan: the planner's answer."""
    _fields_ = [("mode", ctypes.c_int), ("chunk", ctypes.c_int64), ("weight_bytes", ctypes.c_int64),
                ("f16_cache_bytes", ctypes.c_int64), ("act_bytes_per_row", ctypes.c_int64),
                ("total_bytes", ctypes.c_int64)]


class QPGemmDesc(ctypes.Structure):
    """qp_gemm_desc: one projection of a grouped call."""
    _fields_ = [("W", ctypes.c_void_p), ("out_f", ctypes.c_int64), ("in_f", ctypes.c_int64),
                ("X", ctypes.c_void_p), ("Y", ctypes.c_void_p)]

_lib = None


class QPError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, status_str(status), status))


def load():
    """Build (if stale) and load libqp.so; raises if it cannot.  QP_LIBRARY
    names another build of the same sources to load instead."""
    global _lib
    if _lib is None:
        path = os.environ.get("QP_LIBRARY") or _build.build()
        lib = ctypes.CDLL(path)
        i, i64, u64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p
        lib.qp_status_str.argtypes = [i]
        lib.qp_status_str.restype = ctypes.c_char_p
        lib.qp_block_info.argtypes = [i, ctypes.POINTER(i64), ctypes.POINTER(i64)]
        lib.qp_block_info.restype = i
        lib.qp_row_bytes.argtypes = [i, i64]
        lib.qp_row_bytes.restype = i64
        lib.qp_dequant_f32.argtypes = [i, vp, i64, i64, vp, vp]
        lib.qp_dequant_f16.argtypes = [i, vp, i64, i64, vp, vp]
        lib.qp_prefill_gemm.argtypes = [i, vp, i64, i64, vp, i64, vp, vp]
        lib.qp_prefill_gemm_f16w.argtypes = [vp, i64, i64, vp, i64, vp, vp]
        lib.qp_prefill_gemm_group.argtypes = [i, ctypes.POINTER(QPGemmDesc), i, i64, vp]
        lib.qp_prefill_chunked_group.argtypes = [i, ctypes.POINTER(QPGemmDesc), i, i64, i64, vp]
        lib.qp_prefill_chunked.argtypes = [i, vp, vp, i64, i64, vp, i64, vp, i64, i, vp]
        lib.qp_plan_prefill.argtypes = [ctypes.POINTER(QPProjShape), i, i64, i64, i64, i64, i64,
                                        ctypes.POINTER(QPPrefillPlan)]
        lib.qp_decode_gemv.argtypes = [i, vp, i64, i64, vp, i64, vp, vp]
        lib.qp_decode_gemv_group.argtypes = [i, ctypes.POINTER(QPGemmDesc), i, i64, vp]
        lib.qp_check.argtypes = [vp]
        lib.qp_set_wait_limit_ns.argtypes = [u64]
        lib.qp_set_wait_limit_ns.restype = None
        lib.qp_debug_inject_stall.argtypes = [i]
        lib.qp_debug_inject_stall.restype = None
        lib.qp_set_gemm_cta_pairs.argtypes = [i]
        lib.qp_set_gemm_cta_pairs.restype = None
        for name in ("qp_dequant_f32", "qp_dequant_f16", "qp_prefill_gemm", "qp_prefill_gemm_f16w",
                     "qp_prefill_gemm_group", "qp_prefill_chunked_group", "qp_prefill_chunked", "qp_plan_prefill",
                     "qp_decode_gemv", "qp_decode_gemv_group", "qp_check"):
            getattr(lib, name).restype = i
        _lib = lib
    return _lib


def library_path():
    return os.environ.get("QP_LIBRARY") or _build.LIB


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _ok(status, where):
    if status != QP_OK:
        raise QPError(status, where)


def status_str(status):
    return load().qp_status_str(status).decode()


def qp_status_str(status):
    return status_str(status)


def qp_block_info(qtype):
    qk, bb = ctypes.c_int64(), ctypes.c_int64()
    _ok(load().qp_block_info(qtype, ctypes.byref(qk), ctypes.byref(bb)), "qp_block_info")
    return qk.value, bb.value


def qp_row_bytes(qtype, cols):
    return int(load().qp_row_bytes(qtype, cols))


def qp_dequant_f32(qtype, blocks, rows, cols, out, stream=None):
    _ok(load().qp_dequant_f32(qtype, _ptr(blocks), rows, cols, _ptr(out), _stream(stream)), "qp_dequant_f32")


def qp_dequant_f16(qtype, blocks, rows, cols, out, stream=None):
    _ok(load().qp_dequant_f16(qtype, _ptr(blocks), rows, cols, _ptr(out), _stream(stream)), "qp_dequant_f16")


def qp_prefill_gemm(qtype, W, out_f, in_f, X, T, Y, stream=None):
    _ok(load().qp_prefill_gemm(qtype, _ptr(W), out_f, in_f, _ptr(X), T, _ptr(Y), _stream(stream)),
        "qp_prefill_gemm")


def qp_prefill_gemm_f16w(W16, out_f, in_f, X, T, Y, stream=None):
    _ok(load().qp_prefill_gemm_f16w(_ptr(W16), out_f, in_f, _ptr(X), T, _ptr(Y), _stream(stream)),
        "qp_prefill_gemm_f16w")


def _descs(descs):
    arr = (QPGemmDesc * max(len(descs), 1))()
    for k, (W, out_f, in_f, X, Y) in enumerate(descs):
        arr[k] = QPGemmDesc(_ptr(W), out_f, in_f, _ptr(X), _ptr(Y))
    return arr


def qp_prefill_gemm_group(qtype, descs, T, stream=None):
    """descs: sequence of (W, out_f, in_f, X, Y); qtype 0 = fp16 weights (cached mode)."""
    _ok(load().qp_prefill_gemm_group(qtype, _descs(descs), len(descs), T, _stream(stream)),
        "qp_prefill_gemm_group")


def qp_prefill_chunked_group(qtype, descs, T, chunk, stream=None):
    _ok(load().qp_prefill_chunked_group(qtype, _descs(descs), len(descs), T, chunk, _stream(stream)),
        "qp_prefill_chunked_group")


def qp_prefill_chunked(qtype, W, W16, out_f, in_f, X, T, Y, chunk, mode, stream=None):
    _ok(load().qp_prefill_chunked(qtype, _ptr(W), _ptr(W16), out_f, in_f, _ptr(X), T, _ptr(Y), chunk, mode,
                                  _stream(stream)), "qp_prefill_chunked")


def qp_decode_gemv(qtype, W, out_f, in_f, X, T, Y, stream=None):
    _ok(load().qp_decode_gemv(qtype, _ptr(W), out_f, in_f, _ptr(X), T, _ptr(Y), _stream(stream)),
        "qp_decode_gemv")


def qp_decode_gemv_group(qtype, descs, T, stream=None):
    """descs: sequence of (W, out_f, in_f, X, Y), all of type qtype."""
    _ok(load().qp_decode_gemv_group(qtype, _descs(descs), len(descs), T, _stream(stream)), "qp_decode_gemv_group")


def qp_plan_prefill(shapes, T, free_bytes, kv_bytes=0, reserve_bytes=0, max_chunk=0):
    """shapes: sequence of (type, out_f, in_f).  Returns a dict of the plan."""
    arr = (QPProjShape * max(len(shapes), 1))()
    for k, (t, o, i_) in enumerate(shapes):
        arr[k] = QPProjShape(t, o, i_)
    plan = QPPrefillPlan()
    _ok(load().qp_plan_prefill(arr, len(shapes), T, free_bytes, kv_bytes, reserve_bytes, max_chunk,
                               ctypes.byref(plan)), "qp_plan_prefill")
    return {f: getattr(plan, f) for f, _ in QPPrefillPlan._fields_}


def qp_check(stream=None):
    _ok(load().qp_check(_stream(stream)), "qp_check")


def qp_set_wait_limit_ns(ns):
    load().qp_set_wait_limit_ns(int(ns))


def qp_debug_inject_stall(load_index):
    load().qp_debug_inject_stall(int(load_index))


def qp_set_gemm_cta_pairs(on):
    load().qp_set_gemm_cta_pairs(1 if on else 0)
