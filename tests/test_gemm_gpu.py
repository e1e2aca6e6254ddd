"""GPU parity of the batched-prefill projection against the CPU oracle.

Bar (the projection over block-quantized weights, "QK-norm models take the
FP16 batched prefill when it fits", §What changes, with weights from the
per-type dequant of "Qwen3.5 batched prefill has no f32 dequant for IQ2_XXS,
IQ3_S, IQ3_XXS, Q2_K", §Cause): relative Frobenius error <= 1e-3 and
|y - y_ref| <= 4e-3 * sum_k |x||w| elementwise against the fp64 oracle over
the f32 dequantized weight.  Sharper checks that hold by construction:
one-hot X reproduces the f16 weight exactly, fused == cached-f16 bitwise,
chunked == unchunked bitwise, run-to-run determinism, no stray writes.
The full-size workloads are checked in test_gemm_fullsize_gpu.py.
"""
import numpy as np
import pytest

import block_quantized_weight_qp_gb300 as qp
import oracle
import synth
from synth import workloads
from qp_testutil import assert_gemm_within_tolerance, dev, gemm_errors, guard_intact, guarded

pytestmark = pytest.mark.gpu


def torch():
    import torch as t
    return t


@pytest.fixture(params=[1, 0], ids=["cta_pairs", "one_cta"])
def tiling(request):
    """Runs the test on both GEMM tilings: CTA pairs (256-row tiles, the
    default) and one CTA per 128-row tile."""
    qp.qp_set_gemm_cta_pairs(request.param)
    yield request.param
    qp.qp_set_gemm_cta_pairs(1)


def run_gemm(qtype, Wd, out_f, in_f, Xd, T, mode="fused", W16=None, chunk=None):
    t = torch()
    Y = t.empty((T, out_f), dtype=t.float32, device="cuda")
    if chunk is not None:
        qp.qp_prefill_chunked(qtype, Wd, W16, out_f, in_f, Xd, T, Y, chunk, 0 if mode == "fused" else 1)
    elif mode == "fused":
        qp.qp_prefill_gemm(qtype, Wd, out_f, in_f, Xd, T, Y)
    else:
        qp.qp_prefill_gemm_f16w(W16, out_f, in_f, Xd, T, Y)
    qp.qp_check()
    return Y


def dequant16_dev(qtype, Wd, out_f, in_f):
    t = torch()
    W16 = t.empty((out_f, in_f), dtype=t.float16, device="cuda")
    qp.qp_dequant_f16(qtype, Wd, out_f, in_f, W16)
    return W16


def check_against_oracle(qtype, w, X, Y, rows=None, what=""):
    out_f = w.shape[0]
    in_f = X.shape[1]
    W = oracle.dequant_f32(qtype, w, out_f, in_f)
    Yref, A = oracle.gemm_f64(X, W, rows)
    Yg = Y if rows is None else Y[rows]
    rel, ratio = assert_gemm_within_tolerance(Yg, Yref, A, what)
    # diagnostic: against the f16-rounded weights the error is accumulation only
    W16 = W.astype(np.float16).astype(np.float32)
    Yref16, A16 = oracle.gemm_f64(X, W16, rows)
    rel16, _ = gemm_errors(Yg, Yref16, A16)
    assert rel16 <= 2e-5, "%s: error vs f16-rounded-weight reference %.3g" % (what, rel16)
    return rel, ratio, rel16


SMALL = [
    (qp.Q8_0, 256, 512, 16),       # the Q8_0 tiny workload's shape
    (qp.Q4_K, 384, 512, 300),      # 3 weight tiles, ragged token tail
    (qp.Q2_K, 256, 1024, 513),
    (qp.Q6_K, 128, 2048, 77),
    (qp.Q8_0, 640, 768, 1000),
    (qp.Q4_K, 132, 256, 1),        # partial weight tile, one token
    (qp.Q4_K, 4, 256, 3),
    (qp.Q2_K, 1028, 1024, 260),
    (qp.Q5_K, 384, 512, 300),
    (qp.Q5_K, 132, 2048, 77),
    (qp.F16, 260, 512, 129),       # fp16 weights: the cached-mode kernel
]


@pytest.mark.parametrize("qtype,out_f,in_f,T", SMALL, ids=lambda x: str(x))
def test_gemm_small_shapes_vs_oracle(cuda_device, tiling, qtype, out_f, in_f, T):
    w = synth.blocks(qtype, out_f, in_f, seed=out_f + T, tensor=qtype)
    X = synth.normal_f16((T, in_f), seed=out_f + T, tensor=100)
    Y = run_gemm(qtype, dev(w), out_f, in_f, dev(X), T).cpu().numpy()
    check_against_oracle(qtype, w, X, Y, what="%d %dx%d T=%d" % (qtype, out_f, in_f, T))


def test_gemm_q8_0_tiny_workload(cuda_device):
    wl = workloads.WORKLOADS["q8_0_tiny"]
    (_, out_f, in_f, _, qtype), = wl["projections"]
    w = synth.blocks(qtype, out_f, in_f, seed=wl["seed"], tensor=0)
    X = synth.normal_f16((wl["T"], in_f), seed=wl["seed"], tensor=1)
    Y = run_gemm(qtype, dev(w), out_f, in_f, dev(X), wl["T"]).cpu().numpy()
    check_against_oracle(qtype, w, X, Y, what="q8_0_tiny")


@pytest.mark.parametrize("qtype", [qp.Q8_0, qp.Q2_K, qp.Q4_K, qp.Q5_K, qp.Q6_K, qp.F16])
def test_one_hot_rows_reproduce_f16_weights_exactly(cuda_device, tiling, qtype):
    out_f, in_f = 256, 2048
    w = synth.blocks(qtype, out_f, in_f, seed=5, tensor=qtype)
    ks = [0, 1, 15, 16, 31, 32, 63, 64, 100, 127, 128, 255, 256, 511, 1000, 1023, 1024, 2047]
    X = np.zeros((len(ks), in_f), np.float16)
    for t_, k in enumerate(ks):
        X[t_, k] = 1.0
    Y = run_gemm(qtype, dev(w), out_f, in_f, dev(X), len(ks)).cpu().numpy()
    W16 = oracle.dequant_f16(qtype, w, out_f, in_f).view(np.float16).astype(np.float32)
    for t_, k in enumerate(ks):
        assert np.array_equal(Y[t_], W16[:, k]), k


@pytest.mark.parametrize("qtype", [qp.Q8_0, qp.Q2_K, qp.Q4_K, qp.Q5_K, qp.Q6_K, qp.F16])
def test_fused_equals_cached_f16_bitwise(cuda_device, tiling, qtype):
    out_f, in_f, T = 384, 2048, 600
    w = synth.blocks(qtype, out_f, in_f, seed=6, tensor=qtype)
    X = synth.normal_f16((T, in_f), seed=6, tensor=1)
    Wd, Xd = dev(w), dev(X)
    W16 = dequant16_dev(qtype, Wd, out_f, in_f)
    Yf = run_gemm(qtype, Wd, out_f, in_f, Xd, T)
    Yc = run_gemm(qtype, None, out_f, in_f, Xd, T, mode="cached", W16=W16)
    assert torch().equal(Yf.view(torch().int32), Yc.view(torch().int32))


@pytest.mark.parametrize("qtype", [qp.Q8_0, qp.Q2_K, qp.Q4_K, qp.Q5_K, qp.Q6_K, qp.F16])
def test_cta_pair_and_one_cta_tilings_agree_bitwise(cuda_device, qtype):
    """Both tilings run every output through the same K steps of 64 (four
    K = 16 MMAs each, in order) into an fp32 accumulator; only the number of
    weight rows per MMA differs (256 across two SMs, or 128).  Shapes cover a
    pair tile whose second CTA holds no weight rows (out_f = 132, 4) and
    ragged token tails."""
    t = torch()
    in_f = 2048                       # a row of every type is a whole number of 16-byte units
    for out_f, T in ((384, 300), (132, 77), (4, 3), (1028, 513)):
        w = synth.blocks(qtype, out_f, in_f, seed=out_f + 7, tensor=qtype)
        X = synth.normal_f16((T, in_f), seed=out_f + 7, tensor=1)
        Wd, Xd = dev(w), dev(X)
        try:
            qp.qp_set_gemm_cta_pairs(0)
            Y1 = run_gemm(qtype, Wd, out_f, in_f, Xd, T)
        finally:
            qp.qp_set_gemm_cta_pairs(1)
        Y2 = run_gemm(qtype, Wd, out_f, in_f, Xd, T)
        assert t.equal(Y1.view(t.int32), Y2.view(t.int32)), (out_f, in_f, T)


@pytest.mark.parametrize("mode", ["fused", "cached"])
def test_chunked_equals_unchunked_bitwise(cuda_device, mode):
    qtype, out_f, in_f, T = qp.Q4_K, 256, 1024, 1000
    w = synth.blocks(qtype, out_f, in_f, seed=7, tensor=1)
    X = synth.normal_f16((T, in_f), seed=7, tensor=2)
    Wd, Xd = dev(w), dev(X)
    W16 = dequant16_dev(qtype, Wd, out_f, in_f) if mode == "cached" else None
    Y = run_gemm(qtype, Wd, out_f, in_f, Xd, T, mode=mode, W16=W16)
    for chunk in (1000, 999, 256, 300, 77, 1):
        if chunk == 1:
            Xs = Xd[:20]
            Yc = run_gemm(qtype, Wd, out_f, in_f, Xs, 20, mode=mode, W16=W16, chunk=1)
            assert torch().equal(Yc.view(torch().int32), Y[:20].view(torch().int32))
            continue
        Yc = run_gemm(qtype, Wd, out_f, in_f, Xd, T, mode=mode, W16=W16, chunk=chunk)
        assert torch().equal(Yc.view(torch().int32), Y.view(torch().int32)), chunk


GROUP_SHAPES = [(384, 512), (132, 1024), (1028, 256), (4, 512), (256, 2048), (640, 4096), (132, 2048)]


@pytest.mark.parametrize("qtype", [qp.Q8_0, qp.Q2_K, qp.Q4_K, qp.Q5_K, qp.Q6_K, qp.F16])
def test_grouped_launch_equals_single_calls_bitwise(cuda_device, qtype):
    """One persistent launch over several projections (different out_f and
    in_f, each with its own X) gives each Y bitwise as its own call does."""
    t = torch()
    T = 300
    shapes = [(o, i) for o, i in GROUP_SHAPES if qp.qp_row_bytes(qtype, i) % 16 == 0]
    ws = [dev(synth.blocks(qtype, o, i, seed=8, tensor=k)) for k, (o, i) in enumerate(shapes)]
    Xs = [dev(synth.normal_f16((T, i), seed=8, tensor=50 + k)) for k, (o, i) in enumerate(shapes)]
    Ys = [t.full((T, o), float("nan"), dtype=t.float32, device="cuda") for o, i in shapes]
    qp.qp_prefill_gemm_group(qtype, [(w, o, i, X, Y) for w, (o, i), X, Y in zip(ws, shapes, Xs, Ys)], T)
    qp.qp_check()
    assert len(shapes) >= 3
    for w, (o, i), X, Y in zip(ws, shapes, Xs, Ys):
        Y1 = run_gemm(qtype, w, o, i, X, T)
        assert t.equal(Y.view(t.int32), Y1.view(t.int32)), (o, i)


def test_grouped_launch_cached_mode_and_group_limit(cuda_device):
    """type 0 runs the cached mode; eight projections (the limit) in one launch."""
    t = torch()
    qtype, T = qp.Q4_K, 513
    shapes = [(256, 256), (128, 512), (512, 256), (4, 1024), (132, 256), (256, 768), (640, 256), (128, 256)]
    ws = [dev(synth.blocks(qtype, o, i, seed=9, tensor=k)) for k, (o, i) in enumerate(shapes)]
    W16s = [dequant16_dev(qtype, w, o, i) for w, (o, i) in zip(ws, shapes)]
    Xs = [dev(synth.normal_f16((T, i), seed=9, tensor=60 + k)) for k, (o, i) in enumerate(shapes)]
    Yf = [t.empty((T, o), dtype=t.float32, device="cuda") for o, i in shapes]
    Yc = [t.empty((T, o), dtype=t.float32, device="cuda") for o, i in shapes]
    qp.qp_prefill_gemm_group(qtype, [(w, o, i, X, Y) for w, (o, i), X, Y in zip(ws, shapes, Xs, Yf)], T)
    qp.qp_prefill_gemm_group(0, [(w, o, i, X, Y) for w, (o, i), X, Y in zip(W16s, shapes, Xs, Yc)], T)
    qp.qp_check()
    for w, W16, (o, i), X, A, B in zip(ws, W16s, shapes, Xs, Yf, Yc):
        Y1 = run_gemm(qtype, None, o, i, X, T, mode="cached", W16=W16)
        assert t.equal(B.view(t.int32), Y1.view(t.int32)), (o, i)
        assert t.equal(A.view(t.int32), B.view(t.int32)), (o, i)   # fused == cached
    with pytest.raises(qp.QPError):
        qp.qp_prefill_gemm_group(qtype, [(ws[0], 256, 256, Xs[0], Yf[0])] * 9, T)


@pytest.mark.parametrize("mode", ["fused", "cached"])
def test_chunked_group_equals_unchunked_group_bitwise(cuda_device, mode):
    t = torch()
    qtype, T = qp.Q2_K, 777
    shapes = [(256, 1024), (132, 2048), (512, 1024)]
    ws = [dev(synth.blocks(qtype, o, i, seed=10, tensor=k)) for k, (o, i) in enumerate(shapes)]
    if mode == "cached":
        ws = [dequant16_dev(qtype, w, o, i) for w, (o, i) in zip(ws, shapes)]
    ty = qtype if mode == "fused" else 0
    Xs = [dev(synth.normal_f16((T, i), seed=10, tensor=70 + k)) for k, (o, i) in enumerate(shapes)]
    Y = [t.empty((T, o), dtype=t.float32, device="cuda") for o, i in shapes]
    qp.qp_prefill_gemm_group(ty, [(w, o, i, X, y) for w, (o, i), X, y in zip(ws, shapes, Xs, Y)], T)
    for chunk in (777, 256, 300, 1000):
        Yc = [t.full((T, o), float("nan"), dtype=t.float32, device="cuda") for o, i in shapes]
        qp.qp_prefill_chunked_group(ty, [(w, o, i, X, y) for w, (o, i), X, y in zip(ws, shapes, Xs, Yc)], T, chunk)
        qp.qp_check()
        for a, b in zip(Y, Yc):
            assert t.equal(a.view(t.int32), b.view(t.int32)), chunk


def test_deterministic_and_no_stray_writes(cuda_device):
    t = torch()
    qtype, out_f, in_f, T = qp.Q6_K, 260, 2048, 333
    w = synth.blocks(qtype, out_f, in_f, seed=8, tensor=1)
    X = synth.normal_f16((T, in_f), seed=8, tensor=2)
    Wd, Xd = dev(w), dev(X)
    n = T * out_f
    outs = []
    for _ in range(3):
        buf, Y, g = guarded(n, t.float32, out_f)
        qp.qp_prefill_gemm(qtype, Wd, out_f, in_f, Xd, T, Y)
        qp.qp_check()
        assert guard_intact(buf, g, n)
        assert not t.isnan(Y).any()
        outs.append(Y.clone())
    assert t.equal(outs[0].view(t.int32), outs[1].view(t.int32))
    assert t.equal(outs[0].view(t.int32), outs[2].view(t.int32))


@pytest.mark.parametrize("out_f,T,stall", [(256, 300, 5), (1024, 10240, 41)],
                         ids=["first_tile", "third_tile"])
def test_bounded_wait_reports_timeout_and_recovers(cuda_device, tiling, out_f, T, stall):
    """A stage whose copy is never issued: the waits run out after the limit,
    the kernel records the timeout, waits for the copies and MMAs it did
    issue, frees its TMEM and returns; the next call runs normally in the
    same context.  Load `stall` (counted per CTA, 16 loads per tile here)
    falls in the first tile of each CTA, or in the middle of the third tile of
    the CTAs that get three, while the epilogue still drains the second."""
    qtype, in_f = qp.Q4_K, 1024
    w = synth.blocks(qtype, out_f, in_f, seed=9, tensor=1)
    X = synth.normal_f16((T, in_f), seed=9, tensor=2)
    Wd, Xd = dev(w), dev(X)
    t = torch()
    Yok = run_gemm(qtype, Wd, out_f, in_f, Xd, T)
    qp.qp_set_wait_limit_ns(50_000_000)     # 50 ms
    try:
        for mode in ("fused", "cached"):
            W16 = dequant16_dev(qtype, Wd, out_f, in_f) if mode == "cached" else None
            Y = t.empty((T, out_f), dtype=t.float32, device="cuda")
            qp.qp_debug_inject_stall(stall)
            if mode == "fused":
                qp.qp_prefill_gemm(qtype, Wd, out_f, in_f, Xd, T, Y)
            else:
                qp.qp_prefill_gemm_f16w(W16, out_f, in_f, Xd, T, Y)
            with pytest.raises(qp.QPError) as e:
                qp.qp_check()
            assert e.value.status == qp.QP_ERR_TIMEOUT
            qp.qp_check()                    # the word was cleared
            Y2 = run_gemm(qtype, Wd, out_f, in_f, Xd, T)
            assert t.equal(Y2.view(t.int32), Yok.view(t.int32))
    finally:
        qp.qp_set_wait_limit_ns(0)
        qp.qp_debug_inject_stall(-1)
