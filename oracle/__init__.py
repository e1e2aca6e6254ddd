"""CPU oracle for block-quantized weight dequantization and the prefill
projection (scalar C in ``qpo.c``, loaded through ctypes).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers; the product library never
imports, links or runs anything here, and this module imports nothing from
the product.

What it computes and why is documented in ``qpo.h``; in short it follows the
per-type dequantize-to-f32 step and the f16 copy built from it ("Qwen3.5
batched prefill has no f32 dequant for IQ2_XXS, IQ3_S, IQ3_XXS, Q2_K",
§Cause) and the fp64 reference of the batched-prefill GEMM over those weights
("QK-norm models take the FP16 batched prefill when it fits", §What changes).
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "qpo.c")]
_HDR = [os.path.join(_HERE, "qpo.h")]
_SO = os.path.join(_HERE, "_build", "libqpo.so")

F16, Q8_0, Q2_K, Q4_K, Q5_K, Q6_K = 1, 8, 10, 12, 13, 14
# values per block, bytes per block
BLOCK = {F16: (1, 2), Q8_0: (32, 34), Q2_K: (256, 84), Q4_K: (256, 144), Q5_K: (256, 176),
         Q6_K: (256, 210)}

_lib = None


def build(force=False):
    """Compile the oracle with gcc (no FMA contraction, no fast-math)."""
    newest = max(os.path.getmtime(p) for p in _SRC + _HDR)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= newest:
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-fopenmp", "-Wall", "-o", tmp] + _SRC + ["-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _SO)
    return _SO


def lib():
    """The compiled oracle.  QPO_LIB names another build of the same source
    (the planted-fault tests load mutated copies that way)."""
    global _lib
    if _lib is None:
        path = os.environ.get("QPO_LIB") or build()
        l = ctypes.CDLL(path)
        i64, u8p = ctypes.c_int64, ctypes.c_void_p
        l.qpo_block_info.argtypes = [ctypes.c_int, ctypes.POINTER(i64), ctypes.POINTER(i64)]
        l.qpo_f16_to_f32.argtypes = [ctypes.c_uint16]
        l.qpo_f16_to_f32.restype = ctypes.c_float
        l.qpo_f32_to_f16.argtypes = [ctypes.c_float]
        l.qpo_f32_to_f16.restype = ctypes.c_uint16
        l.qpo_f16_to_f32_array.argtypes = [u8p, i64, u8p]
        l.qpo_f32_to_f16_array.argtypes = [u8p, i64, u8p]
        l.qpo_decode_value.argtypes = [ctypes.c_int, u8p, ctypes.c_int]
        l.qpo_decode_value.restype = ctypes.c_float
        l.qpo_dequant_f32.argtypes = [ctypes.c_int, u8p, i64, i64, u8p]
        l.qpo_dequant_f16.argtypes = [ctypes.c_int, u8p, i64, i64, u8p]
        l.qpo_gemm_f64.argtypes = [u8p, u8p, i64, i64, i64, u8p, i64, u8p, u8p]
        l.qpo_num_threads.restype = ctypes.c_int
        l.qpo_set_num_threads.argtypes = [ctypes.c_int]
        # one thread per core this process may run on (the affinity mask, which
        # a container or a job scheduler may set below the machine's count)
        try:
            l.qpo_set_num_threads(len(os.sched_getaffinity(0)))
        except (AttributeError, OSError):
            pass
        _lib = l
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads():
    return int(lib().qpo_num_threads())


def set_num_threads(n):
    """Threads of the oracle's OpenMP regions (parallelism only: every output
    value is computed by one thread in a fixed order)."""
    lib().qpo_set_num_threads(int(n))


def f16_to_f32(h):
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().qpo_f16_to_f32_array(_ptr(h), h.size, _ptr(out))
    return out


def f32_to_f16(f):
    """Returns fp16 bit patterns (uint16)."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, np.uint16)
    lib().qpo_f32_to_f16_array(_ptr(f), f.size, _ptr(out))
    return out


def decode_value(qtype, block, v):
    block = np.ascontiguousarray(block, dtype=np.uint8)
    return float(lib().qpo_decode_value(qtype, _ptr(block), int(v)))


def _check_blocks(qtype, blocks, rows, cols):
    qk, bb = BLOCK[qtype]
    nb = -(-cols // qk)
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    if blocks.size != rows * nb * bb:
        raise ValueError("blocks hold %d bytes, expected %d" % (blocks.size, rows * nb * bb))
    return blocks


GUARD = 4096  # elements of NaN guard band after every oracle output


def _guarded(n, dtype, nan_bits):
    buf = np.empty(n + GUARD, dtype)
    buf.view(np.uint32 if dtype == np.float32 else np.uint16)[:] = nan_bits
    return buf


def _check_guard(buf, n, nan_bits):
    tail = buf[n:].view(np.uint32 if buf.dtype == np.float32 else np.uint16)
    if not np.all(tail == nan_bits):
        raise AssertionError("oracle wrote past the end of its output")


def dequant_f32(qtype, blocks, rows, cols):
    blocks = _check_blocks(qtype, blocks, rows, cols)
    buf = _guarded(rows * cols, np.float32, 0x7fc00000)
    if lib().qpo_dequant_f32(qtype, _ptr(blocks), rows, cols, _ptr(buf)):
        raise ValueError("bad type %r" % qtype)
    _check_guard(buf, rows * cols, 0x7fc00000)
    return buf[:rows * cols].reshape(rows, cols)


def dequant_f16(qtype, blocks, rows, cols):
    """Returns fp16 bit patterns (uint16) of shape [rows, cols]."""
    blocks = _check_blocks(qtype, blocks, rows, cols)
    buf = _guarded(rows * cols, np.uint16, 0x7e00)
    if lib().qpo_dequant_f16(qtype, _ptr(blocks), rows, cols, _ptr(buf)):
        raise ValueError("bad type %r" % qtype)
    _check_guard(buf, rows * cols, 0x7e00)
    return buf[:rows * cols].reshape(rows, cols)


def gemm_f64(X, W, rows=None):
    """fp64 reference Y = X W^T and A = |X| |W|^T for the token rows `rows`.

    X: [T, in] fp16 bit patterns (uint16) or float16; W: [out, in] float32.
    Returns (Y, A), each [len(rows), out] float64."""
    X = np.ascontiguousarray(X).view(np.uint16)
    W = np.ascontiguousarray(W, dtype=np.float32)
    T, k = X.shape
    out, k2 = W.shape
    if k != k2:
        raise ValueError("inner dimensions differ")
    if rows is None:
        nrows, rp = T, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        if rows.size and (rows.min() < 0 or rows.max() >= T):
            raise ValueError("row index out of range")
        nrows, rp = rows.size, _ptr(rows)
    Y = np.empty((nrows, out), np.float64)
    A = np.empty((nrows, out), np.float64)
    lib().qpo_gemm_f64(_ptr(X), _ptr(W), T, out, k, rp, nrows, _ptr(Y), _ptr(A))
    return Y, A
