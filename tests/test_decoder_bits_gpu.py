"""The fused GEMM's decoders and the decode GEMV's run decoders on blocks
whose every quant, scale and min byte is random: all bit patterns of every
field occur, among them the int8 value -128 (a Q8_0 quant, a Q6_K scale) and
the top bits of the packed 6-bit Q4_K/Q5_K scales ("Qwen3.5 batched prefill
has no f32 dequant for IQ2_XXS, IQ3_S, IQ3_XXS, Q2_K", §Acceptance: signs,
high bits and the scale selector).  d and dmin stay finite so that every
weight is a finite fp16 number.

- GEMM: X = the identity (T = in_f one-hot token rows) makes Y the transpose
  of the fp16 weight, so every fp16 weight the decoders produce is compared
  with the oracle's, exactly; and random X against the fp64 oracle at the
  workload tolerance.  Both tilings.
- GEMV: one-hot rows over every column of the weight (1, 2, 4 or 8 per
  launch: each token-column layout of the K-quant kernels), exact (the f32
  weights for the K-quants, the fp16 weights for Q8_0), and random X
  against the oracle.
"""
import numpy as np
import pytest

import block_quantized_weight_qp_gb300 as qp
import oracle
import synth
from qp_testutil import assert_gemm_within_tolerance, dev

pytestmark = pytest.mark.gpu

QUANT_TYPES = [qp.Q8_0, qp.Q2_K, qp.Q4_K, qp.Q5_K, qp.Q6_K]
ID = {qp.Q8_0: "Q8_0", qp.Q2_K: "Q2_K", qp.Q4_K: "Q4_K", qp.Q5_K: "Q5_K", qp.Q6_K: "Q6_K"}


def torch():
    import torch as t
    return t


@pytest.fixture(params=[1, 0], ids=["cta_pairs", "one_cta"])
def tiling(request):
    qp.qp_set_gemm_cta_pairs(request.param)
    yield request.param
    qp.qp_set_gemm_cta_pairs(1)


def weights(qtype, out_f, in_f, seed):
    w = synth.blocks_anybits(qtype, out_f, in_f, seed=seed, tensor=qtype)
    bb = oracle.BLOCK[qtype][1]
    blk = w.reshape(-1, bb)
    if qtype == qp.Q8_0:
        assert (blk[:, 2:].view(np.int8) == -128).any()
    if qtype == qp.Q6_K:
        assert (blk[:, 192:208].view(np.int8) == -128).any()
    W16 = oracle.dequant_f16(qtype, w, out_f, in_f).view(np.float16)
    assert np.isfinite(W16).all()
    return w, W16


@pytest.mark.parametrize("qtype", QUANT_TYPES, ids=lambda q: ID[q])
def test_gemm_identity_gives_every_f16_weight(cuda_device, tiling, qtype):
    t = torch()
    out_f, in_f = 260, 2048
    w, W16 = weights(qtype, out_f, in_f, seed=41)
    X = np.eye(in_f, dtype=np.float16)
    Y = t.full((in_f, out_f), float("nan"), dtype=t.float32, device="cuda")
    qp.qp_prefill_gemm(qtype, dev(w), out_f, in_f, dev(X), in_f, Y)
    qp.qp_check()
    got = Y.cpu().numpy()
    # a -0 weight may come out +0 from the sum of signed zeros; compare values
    assert np.array_equal(got, W16.astype(np.float32).T)


@pytest.mark.parametrize("qtype", QUANT_TYPES, ids=lambda q: ID[q])
def test_gemm_random_fields_vs_oracle(cuda_device, tiling, qtype):
    t = torch()
    out_f, in_f, T = 260, 2048, 300
    w, _ = weights(qtype, out_f, in_f, seed=42)
    X = synth.normal_f16((T, in_f), seed=42, tensor=7)
    Y = t.empty((T, out_f), dtype=t.float32, device="cuda")
    qp.qp_prefill_gemm(qtype, dev(w), out_f, in_f, dev(X), T, Y)
    qp.qp_check()
    Yref, A = oracle.gemm_f64(X, oracle.dequant_f32(qtype, w, out_f, in_f))
    assert_gemm_within_tolerance(Y.cpu().numpy(), Yref, A, "random fields %s" % ID[qtype])


@pytest.mark.parametrize("T", [8, 4, 2, 1])
@pytest.mark.parametrize("in_f", [2048, 1280], ids=["tma_tiles", "row_copies"])
@pytest.mark.parametrize("qtype", QUANT_TYPES, ids=lambda q: ID[q])
def test_gemv_one_hot_over_every_column(cuda_device, qtype, in_f, T):
    """Every weight of every row, exactly.  With 1280 values a Q2_K or Q6_K
    row is not a whole number of 16-byte words, so the rows are staged by one
    copy each and (Q6_K) every other row starts 2 bytes past a word.  A -0
    weight comes out +0 (it is added to +0 sums)."""
    t = torch()
    out_f = 72
    w, W16 = weights(qtype, out_f, in_f, seed=43)
    if qtype == qp.Q8_0:
        want = W16.astype(np.float32) + np.float32(0.0)
    else:
        want = oracle.dequant_f32(qtype, w, out_f, in_f) + np.float32(0.0)
    Wd = dev(w)
    n = in_f // T
    X = np.zeros((n, T, in_f), np.float16)
    for j in range(n):
        for r in range(T):
            X[j, r, j * T + r] = 1.0
    Xd = dev(X)
    Y = t.full((n, T, out_f), float("nan"), dtype=t.float32, device="cuda")
    for j in range(n):
        qp.qp_decode_gemv(qtype, Wd, out_f, in_f, Xd[j], T, Y[j])
    qp.qp_check()
    got = Y.cpu().numpy().reshape(in_f, out_f)
    assert np.array_equal(got.view(np.uint32), np.ascontiguousarray(want.T).view(np.uint32))


@pytest.mark.parametrize("qtype", QUANT_TYPES, ids=lambda q: ID[q])
def test_gemv_random_fields_vs_oracle(cuda_device, qtype):
    t = torch()
    out_f, in_f, T = 136, 4096, 5
    w, _ = weights(qtype, out_f, in_f, seed=44)
    X = synth.normal_f16((T, in_f), seed=44, tensor=8)
    Y = t.empty((T, out_f), dtype=t.float32, device="cuda")
    qp.qp_decode_gemv(qtype, dev(w), out_f, in_f, dev(X), T, Y)
    qp.qp_check()
    Yref, A = oracle.gemm_f64(X, oracle.dequant_f32(qtype, w, out_f, in_f))
    assert_gemm_within_tolerance(Y.cpu().numpy(), Yref, A, "gemv random fields %s" % ID[qtype])
