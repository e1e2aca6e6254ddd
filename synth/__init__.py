"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

Only random draws and byte placement live here (``synth.c``): no decoding, no
scale unpacking, no GEMM.  Every tensor is a pure function of (seed, tensor
id), so the oracle side and the GPU side get identical bytes.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "_build", "libqpsynth.so")

F16, Q8_0, Q2_K, Q4_K, Q5_K, Q6_K = 1, 8, 10, 12, 13, 14
# values per block, bytes per block
BLOCK = {F16: (1, 2), Q8_0: (32, 34), Q2_K: (256, 84), Q4_K: (256, 144), Q5_K: (256, 176), Q6_K: (256, 210)}
NAMES = {F16: "F16", Q8_0: "Q8_0", Q2_K: "Q2_K", Q4_K: "Q4_K", Q5_K: "Q5_K", Q6_K: "Q6_K"}

_lib = None


def build(force=False):
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + ".tmp.%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
                           "-Wall", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        l = ctypes.CDLL(build())
        u64, i64, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        l.synth_key.argtypes = [u64, u64]
        l.synth_key.restype = u64
        l.synth_blocks.argtypes = [ctypes.c_int, u64, i64, vp]
        l.synth_blocks_anybits.argtypes = [ctypes.c_int, u64, i64, vp]
        l.synth_normal_f16.argtypes = [u64, i64, vp]
        l.synth_bytes.argtypes = [u64, i64, vp]
        _lib = l
    return _lib


def key(seed, tensor):
    return int(lib().synth_key(seed, tensor))


def row_bytes(qtype, cols):
    qk, bb = BLOCK[qtype]
    return -(-cols // qk) * bb


def blocks(qtype, rows, cols, seed, tensor=0):
    """Row-major [rows, ceil(cols/QK)] blocks as a uint8 array [rows, row_bytes]."""
    qk, bb = BLOCK[qtype]
    nb = -(-cols // qk)
    out = np.empty((rows, nb * bb), np.uint8)
    lib().synth_blocks(qtype, key(seed, tensor), rows * nb, out.ctypes.data_as(ctypes.c_void_p))
    return out


def blocks_anybits(qtype, rows, cols, seed, tensor=0):
    """As ``blocks``, but every quant, scale and min byte is a uniform random
    byte (all bit patterns of every field, int8 -128 included); the fp16 d and
    dmin fields are drawn as in ``blocks``, so every weight stays finite."""
    qk, bb = BLOCK[qtype]
    nb = -(-cols // qk)
    out = np.empty((rows, nb * bb), np.uint8)
    lib().synth_blocks_anybits(qtype, key(seed, tensor), rows * nb, out.ctypes.data_as(ctypes.c_void_p))
    return out


def normal_f16(shape, seed, tensor=0):
    """Standard-normal values on the fp16 grid, as a float16 array."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    lib().synth_normal_f16(key(seed, tensor), n, out.ctypes.data_as(ctypes.c_void_p))
    return out.view(np.float16).reshape(shape)


def random_bytes(n, seed, tensor=0):
    out = np.empty(n, np.uint8)
    lib().synth_bytes(key(seed, tensor), n, out.ctypes.data_as(ctypes.c_void_p))
    return out
