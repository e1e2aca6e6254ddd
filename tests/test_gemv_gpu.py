"""GPU parity of qp_decode_gemv (the decode-side projection over the same
weight blocks, T = 1..8 token rows) against the CPU oracle's fp64
reference: the GEMM tolerance of the workload definition, exact one-hot
rows (the GEMV multiplies the exact f32 weights of qp_dequant_f32 for the
K-quants, and the fp16 weights of qp_dequant_f16 for Q8_0 and F16),
determinism, and every token-column layout of the K-quant kernels."""
import numpy as np
import pytest

import block_quantized_weight_qp_gb300 as qp
import oracle
import synth
from qp_testutil import assert_gemm_within_tolerance, dev

pytestmark = pytest.mark.gpu

CASES = [
    (qp.Q4_K, 384, 4096, 1),
    (qp.Q4_K, 37, 1024, 3),          # a partial warp of rows
    (qp.Q2_K, 256, 4096, 8),
    (qp.Q6_K, 132, 12288, 8),        # long rows: 384 runs over the CTA's warps
    (qp.Q6_K, 64, 2048, 1),
    (qp.Q5_K, 200, 2048, 5),
    (qp.Q8_0, 256, 512, 8),
    (qp.Q8_0, 9, 96, 2),             # three runs per row: most lanes idle
    (qp.F16, 260, 1024, 4),
    (qp.F16, 1, 32, 1),
    (qp.Q2_K, 1029, 1024, 7),        # 65 row blocks of 16, the last with 5 rows
    (qp.F16, 24, 13056, 8),          # 408 runs: a partial last step
    (qp.Q8_0, 16, 4128, 6),          # 129 runs
    (qp.Q2_K, 48, 768, 3),           # rows of 252 bytes: staged by one copy per row
    (qp.Q6_K, 40, 1280, 2),          # rows of 1050 bytes: odd rows start 2 bytes past a word
]


def gemv(qtype, Wd, out_f, in_f, Xd, T):
    import torch
    Y = torch.full((T, out_f), float("nan"), dtype=torch.float32, device="cuda")
    qp.qp_decode_gemv(qtype, Wd, out_f, in_f, Xd, T, Y)
    qp.qp_check()
    return Y


@pytest.mark.parametrize("qtype,out_f,in_f,T", CASES, ids=lambda x: str(x))
def test_decode_gemv_vs_oracle(cuda_device, qtype, out_f, in_f, T):
    w = synth.blocks(qtype, out_f, in_f, seed=out_f + T, tensor=qtype)
    X = synth.normal_f16((T, in_f), seed=out_f + T, tensor=200)
    Y = gemv(qtype, dev(w), out_f, in_f, dev(X), T).cpu().numpy()
    W = oracle.dequant_f32(qtype, w, out_f, in_f)
    Yref, A = oracle.gemm_f64(X, W)
    assert_gemm_within_tolerance(Y, Yref, A, "gemv %d %dx%d T=%d" % (qtype, out_f, in_f, T))


KQUANTS = [qp.Q2_K, qp.Q4_K, qp.Q5_K, qp.Q6_K]


@pytest.mark.parametrize("qtype", [qp.Q8_0, qp.Q2_K, qp.Q4_K, qp.Q5_K, qp.Q6_K, qp.F16])
def test_decode_gemv_one_hot_rows_give_the_weights(cuda_device, qtype):
    """A one-hot X row returns a column of the weights bit for bit: the f32
    dequant for the K-quants (their codes are multiplied as exact fp16
    subnormals and the sub-block scales applied in f32), the fp16 dequant
    for Q8_0 and F16."""
    out_f, in_f = 96, 2048
    w = synth.blocks(qtype, out_f, in_f, seed=13, tensor=qtype)
    if qtype in KQUANTS:
        W = oracle.dequant_f32(qtype, w, out_f, in_f)
    else:
        W = oracle.dequant_f16(qtype, w, out_f, in_f).view(np.float16).astype(np.float32)
    for ks in ([0, 31, 32, 255, 256, 1000, 2047, 1024], [7], [2046, 1], [15, 16, 17], [300, 511, 512, 513, 1535]):
        X = np.zeros((len(ks), in_f), np.float16)
        for t, k in enumerate(ks):
            X[t, k] = 1.0
        Y = gemv(qtype, dev(w), out_f, in_f, dev(X), len(ks)).cpu().numpy()
        for t, k in enumerate(ks):
            # the dot product adds the weight to +0 partial sums: a -0 weight (Q6_K q = 32
            # under a negative scale) comes out +0, as IEEE addition gives
            want = W[:, k] + np.float32(0.0)
            assert np.array_equal(Y[t].view(np.uint32), want.view(np.uint32)), (qtype, k)


@pytest.mark.parametrize("qtype", KQUANTS)
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("out_f,in_f", [(48, 1024), (40, 1280)])
def test_decode_gemv_every_token_layout(cuda_device, qtype, T, out_f, in_f):
    """The K-quant kernels take 8 / T sub-blocks per MMA (T rounded up to a
    power of two): each layout, with TMA-staged rows and, at in_f = 1280,
    Q2_K and Q6_K rows whose pitch is no multiple of 16 bytes (staged row by
    row; Q6_K rows then start 2 bytes past a word every other row)."""
    w = synth.blocks(qtype, out_f, in_f, seed=40 + T, tensor=qtype)
    X = synth.normal_f16((T, in_f), seed=50 + T, tensor=3)
    Y = gemv(qtype, dev(w), out_f, in_f, dev(X), T).cpu().numpy()
    Yref, A = oracle.gemm_f64(X, oracle.dequant_f32(qtype, w, out_f, in_f))
    assert_gemm_within_tolerance(Y, Yref, A, "gemv %d %dx%d T=%d" % (qtype, out_f, in_f, T))


def test_decode_gemv_is_deterministic(cuda_device):
    import torch
    qtype, out_f, in_f, T = qp.Q2_K, 1024, 4096, 8
    Wd = dev(synth.blocks(qtype, out_f, in_f, seed=14, tensor=1))
    Xd = dev(synth.normal_f16((T, in_f), seed=14, tensor=2))
    a = gemv(qtype, Wd, out_f, in_f, Xd, T)
    b = gemv(qtype, Wd, out_f, in_f, Xd, T)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("T", [1, 5])
@pytest.mark.parametrize("qtype", [qp.Q8_0, qp.Q2_K, qp.Q4_K, qp.Q5_K, qp.Q6_K, qp.F16])
def test_grouped_decode_gemv_equals_single_calls_bitwise(cuda_device, qtype, T):
    """One launch over several projections (own X, own Y each, the long-K
    one and a one-superblock one included) gives every Y bitwise as its own
    call does.  T = 1: the K-quant blocks end without a barrier (the warp
    that completes a block's count sums it); T = 5: with one."""
    import torch
    shapes = [(37, 1024), (256, 4096), (8, 2048), (1029, 1024), (64, 12288), (4000, 256)]
    ws = [dev(synth.blocks(qtype, o, i, seed=20 + k, tensor=qtype)) for k, (o, i) in enumerate(shapes)]
    xs = [dev(synth.normal_f16((T, i), seed=30 + k, tensor=1)) for k, (o, i) in enumerate(shapes)]
    singles = [gemv(qtype, w, o, i, x, T) for w, (o, i), x in zip(ws, shapes, xs)]
    ys = [torch.full((T, o), float("nan"), dtype=torch.float32, device="cuda") for o, _ in shapes]
    qp.qp_decode_gemv_group(qtype, [(w, o, i, x, y) for w, (o, i), x, y in zip(ws, shapes, xs, ys)], T)
    qp.qp_check()
    for k, (a, b) in enumerate(zip(singles, ys)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), shapes[k]


@pytest.mark.parametrize("T", [1, 2, 3, 4])
@pytest.mark.parametrize("qtype", KQUANTS)
def test_decode_gemv_many_one_step_blocks_vs_oracle(cuda_device, qtype, T):
    """Rows of one superblock, 16,000 of them: each 16-row block is a single
    one-step tile, so seven of a CTA's eight consumer warps have no step in
    it and run ahead to the ring's depth, and every CTA ends many blocks
    in a row.  Their partial tiles are summed by whichever warp completes a
    block's count, from buffers reused every NST + 1 blocks."""
    out_f, in_f = 16000, 256
    w = synth.blocks(qtype, out_f, in_f, seed=41 + T, tensor=qtype)
    X = synth.normal_f16((T, in_f), seed=41 + T, tensor=7)
    Y = gemv(qtype, dev(w), out_f, in_f, dev(X), T).cpu().numpy()
    W = oracle.dequant_f32(qtype, w, out_f, in_f)
    Yref, A = oracle.gemm_f64(X, W)
    assert_gemm_within_tolerance(Y, Yref, A, "gemv %d %dx%d T=%d" % (qtype, out_f, in_f, T))


@pytest.mark.parametrize("T", [1, 5])
@pytest.mark.parametrize("stall", [1, 6], ids=["prefill_tile", "ring_tile"])
def test_decode_gemv_bounded_wait_reports_timeout_and_recovers(cuda_device, T, stall):
    """A ring tile whose copy is never issued (each CTA's tile `stall`: one
    of the first tiles, which go out one at a time, or one past them): the
    consumers' wait runs out after the limit, the launch records the timeout
    and returns, every warp still ending every block (T = 1: the arrival
    count; T = 5: the named barrier); the next call runs normally in the
    same context and gives the clean result bit for bit.  34,816 Q2_K rows
    (2,176 blocks of one tile each) give each of up to 304 CTAs at least
    seven tiles."""
    import torch
    qtype, out_f, in_f = qp.Q2_K, 34816, 4096
    Wd = dev(synth.blocks(qtype, out_f, in_f, seed=51, tensor=1))
    Xd = dev(synth.normal_f16((T, in_f), seed=51, tensor=2))
    Yok = gemv(qtype, Wd, out_f, in_f, Xd, T)
    qp.qp_set_wait_limit_ns(50_000_000)     # 50 ms
    try:
        Y = torch.full((T, out_f), float("nan"), dtype=torch.float32, device="cuda")
        qp.qp_debug_inject_stall(stall)
        qp.qp_decode_gemv(qtype, Wd, out_f, in_f, Xd, T, Y)
        with pytest.raises(qp.QPError) as e:
            qp.qp_check()
        assert e.value.status == qp.QP_ERR_TIMEOUT
        qp.qp_check()                        # the word was cleared
        Y2 = gemv(qtype, Wd, out_f, in_f, Xd, T)
        assert torch.equal(Y2.view(torch.int32), Yok.view(torch.int32))
    finally:
        qp.qp_set_wait_limit_ns(0)
        qp.qp_debug_inject_stall(-1)


def test_decode_gemv_reads_operands_written_just_before(cuda_device):
    """A GEMV may start while the previous kernel on the stream (one of this
    library's, which let the next launch begin early) still runs.  F16
    weights that qp_dequant_f16 writes right before it are read only after
    that kernel, and so is X: here X is itself the output of a dequant
    launched just before a K-quant GEMV.  Repeated with fresh values, so
    stale data would show."""
    import torch
    out_f, in_f, T = 512, 4096, 1
    for rep in range(3):
        w = synth.blocks(qp.Q4_K, out_f, in_f, seed=60 + rep, tensor=1)
        Wd = dev(w)
        W16 = torch.full((out_f, in_f), float("nan"), dtype=torch.float16, device="cuda")
        X = dev(synth.normal_f16((T, in_f), seed=61 + rep, tensor=2))
        Y1 = torch.full((T, out_f), float("nan"), dtype=torch.float32, device="cuda")
        qp.qp_dequant_f16(qp.Q4_K, Wd, out_f, in_f, W16)
        qp.qp_decode_gemv(qp.F16, W16, out_f, in_f, X, T, Y1)
        # X of the next GEMV: a 1 x 512 Q4_K tensor dequantized right before it
        xq = synth.blocks(qp.Q4_K, T, out_f, seed=62 + rep, tensor=3)
        X2 = torch.full((T, out_f), float("nan"), dtype=torch.float16, device="cuda")
        w2 = synth.blocks(qp.Q2_K, 256, out_f, seed=63 + rep, tensor=4)
        W2d = dev(w2)
        Y2 = torch.full((T, 256), float("nan"), dtype=torch.float32, device="cuda")
        qp.qp_dequant_f16(qp.Q4_K, dev(xq), T, out_f, X2)
        qp.qp_decode_gemv(qp.Q2_K, W2d, 256, out_f, X2, T, Y2)
        qp.qp_check()
        Wf = oracle.dequant_f16(qp.Q4_K, w, out_f, in_f).view(np.float16).astype(np.float32)
        Yref, A = oracle.gemm_f64(X.cpu().numpy(), Wf)
        assert_gemm_within_tolerance(Y1.cpu().numpy(), Yref, A, "F16 GEMV after the dequant of its weights")
        X2ref = oracle.dequant_f16(qp.Q4_K, xq, T, out_f).view(np.float16)
        assert np.array_equal(X2.cpu().numpy().view(np.uint16), X2ref.view(np.uint16))
        Y2ref, A2 = oracle.gemm_f64(X2ref, oracle.dequant_f32(qp.Q2_K, w2, 256, out_f))
        assert_gemm_within_tolerance(Y2.cpu().numpy(), Y2ref, A2, "Q2_K GEMV after the dequant of its X")
