"""The arithmetic the decode GEMV rests on, checked on the CPU against the
oracle.  For the K-quants the GEMV multiplies raw codes u and applies, per
sub-block of a row, w = alpha * (u * 2^-24) + beta, with

  Q2_K, Q4_K, Q5_K: alpha = d * sc * 2^24, beta = -(dmin * m)
  Q6_K:             alpha = d * s * 2^24,  beta = -32 * d * s

(the value formulas of the K-quant page, "Q2_K", "Q4_K", "Q5_K" and "Q6_K"
sections, written as affine functions of the code).  If alpha and beta are
exact in f32 and alpha * u * 2^-24 + beta is rounded once, the result must
be the oracle's f32 dequant bit for bit, for every value of every block;
random field bytes reach every scale, min and code (d and dmin in their
workload range, so the fp64 sum below is exact and its conversion to f32 is
the single rounding).  The fields are parsed here from the block bytes,
independently of the oracle's C decoder.
"""
import numpy as np
import pytest

import oracle
import synth

Q2_K, Q4_K, Q5_K, Q6_K = oracle.Q2_K, oracle.Q4_K, oracle.Q5_K, oracle.Q6_K


def h(b, o):
    return float(np.frombuffer(bytes(b[o:o + 2]), np.float16)[0])


def k4_scale_min(sc12, s):
    """6-bit (sc, m) of sub-block s from the 12 packed scale bytes."""
    if s < 4:
        return sc12[s] & 63, sc12[s + 4] & 63
    return ((sc12[s + 4] & 15) | ((sc12[s - 4] >> 6) << 4),
            (sc12[s + 4] >> 4) | ((sc12[s] >> 6) << 4))


def affine_fields(qtype, b):
    """Per value v of one superblock: (code u, alpha, beta) as exact floats."""
    out = []
    for v in range(256):
        if qtype == Q2_K:
            n, j, l, s = v // 128, (v % 128) // 32, v % 32, v // 16
            u = (b[16 + 32 * n + l] >> (2 * j)) & 3
            d, dmin = h(b, 80), h(b, 82)
            alpha, beta = d * (b[s] & 15) * 2.0 ** 24, -(dmin * (b[s] >> 4))
        elif qtype == Q6_K:
            n, j, l, s = v // 128, (v % 128) // 32, v % 32, v // 16
            qlb = b[64 * n + 32 * (j & 1) + l]
            lo = (qlb >> 4) if j >= 2 else (qlb & 15)
            u = lo | (((b[128 + 32 * n + l] >> (2 * j)) & 3) << 4)
            sv = int(np.int8(np.uint8(b[192 + s])))
            d = h(b, 208)
            alpha, beta = d * sv * 2.0 ** 24, -32.0 * d * sv
        else:
            q5 = qtype == Q5_K
            s, l = v // 32, v % 32
            qs = 48 if q5 else 16
            byte = b[qs + 32 * (s // 2) + l]
            u = (byte >> 4) if s % 2 else (byte & 15)
            if q5:
                u |= ((b[16 + l] >> s) & 1) << 4
            sc, m = k4_scale_min(b[4:16], s)
            d, dmin = h(b, 0), h(b, 2)
            alpha, beta = d * sc * 2.0 ** 24, -(dmin * m)
        out.append((u, alpha, beta))
    return out


@pytest.mark.parametrize("qtype", [Q2_K, Q4_K, Q5_K, Q6_K], ids=["Q2_K", "Q4_K", "Q5_K", "Q6_K"])
def test_k_quant_weights_are_affine_in_the_code_with_exact_factors(qtype):
    rows, cols = 6, 1024
    w = synth.blocks_anybits(qtype, rows, cols, seed=71, tensor=qtype)
    ref = oracle.dequant_f32(qtype, w, rows, cols)
    bb = oracle.BLOCK[qtype][1]
    blocks = w.reshape(rows, -1, bb)
    for r in range(rows):
        for k in range(cols // 256):
            for v, (u, alpha, beta) in enumerate(affine_fields(qtype, blocks[r, k])):
                # the factors are exact f32 numbers
                assert np.float32(alpha) == alpha and np.float32(beta) == beta
                code = u * 2.0 ** -24                 # the fp16 subnormal field, exactly
                assert float(np.array([u], np.uint16).view(np.float16)[0]) == code
                # one rounding of the exact value (alpha * code is exact in fp64 here)
                got = np.float32(alpha * code + beta)
                want = ref[r, 256 * k + v]
                assert got.view(np.uint32) == np.float32(want).view(np.uint32) or (got == 0 and want == 0), \
                    (r, k, v, u, alpha, beta, got, want)
