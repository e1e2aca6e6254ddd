"""Full-size parity of the batched-prefill projection against the fp64 CPU
oracle, on the layer workloads and in the launch configuration the benchmark
times.

The bar ("Qwen3.5 batched prefill has no f32 dequant for IQ2_XXS, IQ3_S,
IQ3_XXS, Q2_K", §Acceptance: every tensor checked, not samples; the workload
tolerance): relative Frobenius error <= 1e-3 over each projection's whole
output and |y - y_ref| <= 4e-3 * sum_k |x||w| for every element.

- The Qwen3-1.7B-shaped Q4_K layer (T = 2048) and the Qwen3-8B-shaped
  Q2_K/Q6_K layer (T = 8192): every element of all seven outputs, issued as
  one grouped launch per run of projections of one block type ("QK-norm
  models take the FP16 batched prefill when it fits", §What changes: one GEMM
  per projection over the prompt chunk).
- The 31,258-token prompt in chunks of 4,864 ("CUDA prefill VRAM loans and
  SM75 Q4/native-IQ opt-ins", §End-to-end results: the 4,864-token prompt
  chunk) through the 8B-shaped Q4_K layer, issued as the benchmark issues it
  (one grouped launch per chunk): all seven projections at both rows of every
  chunk boundary, the last row and every 16th row; fused-chunked ==
  fused-unchunked == cached-f16-chunked bitwise over whole outputs.

The oracle runs in row blocks so that its fp64 outputs stay small.
"""
import numpy as np
import pytest

import block_quantized_weight_qp_gb300 as qp
import oracle
import synth
from synth import workloads
from qp_testutil import GemmErrorTally, dev


def torch():
    import torch as t
    return t


def layer_inputs(wl):
    dims = workloads.input_dims(wl)
    return {k: synth.normal_f16((wl["T"], dims[k]), seed=wl["seed"], tensor=1000 + i)
            for i, k in enumerate(("h", "o", "f"))}


def issue_layer(wl, Wd, Xd, Y, chunk=None, W16=None):
    """The layer's projections as the benchmark issues them: one grouped
    launch (or one chunked grouped call) per run of one block type."""
    for qt, idx in workloads.type_runs(wl["projections"]):
        descs = []
        for i in idx:
            _, out_f, in_f, src, _ = wl["projections"][i]
            descs.append((Wd[i] if W16 is None else W16[i], out_f, in_f, Xd[src], Y[i]))
        ty = qt if W16 is None else 0
        if chunk:
            qp.qp_prefill_chunked_group(ty, descs, wl["T"], chunk)
        else:
            qp.qp_prefill_gemm_group(ty, descs, wl["T"])
    qp.qp_check()


def check_rows(Yd, X, W32, rows, what, block=1024):
    """Y[rows] of one projection against the fp64 oracle, `block` rows at a time."""
    t = torch()
    tally = GemmErrorTally(what)
    for i in range(0, rows.size, block):
        r = rows[i:i + block]
        Yref, A = oracle.gemm_f64(X, W32, r)
        Yg = Yd.index_select(0, t.from_numpy(r).to(Yd.device)).cpu().numpy()
        tally.add(Yg, Yref, A)
    return tally.check()


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["qwen3_1p7b_q4k_t2048", "qwen3_8b_q2k_q6k_t8192"])
def test_full_size_layer_every_output_vs_oracle(cuda_device, name):
    t = torch()
    wl = workloads.WORKLOADS[name]
    T = wl["T"]
    X = layer_inputs(wl)
    Xd = {k: dev(v) for k, v in X.items()}
    W = [synth.blocks(qt, out_f, in_f, seed=wl["seed"], tensor=i)
         for i, (_, out_f, in_f, _, qt) in enumerate(wl["projections"])]
    Wd = [dev(w) for w in W]
    Y = [t.full((T, out_f), float("nan"), dtype=t.float32, device="cuda")
         for (_, out_f, _, _, _) in wl["projections"]]
    issue_layer(wl, Wd, Xd, Y)
    rows = np.arange(T, dtype=np.int64)
    for i, (pname, out_f, in_f, src, qt) in enumerate(wl["projections"]):
        W32 = oracle.dequant_f32(qt, W[i], out_f, in_f)
        check_rows(Y[i], X[src], W32, rows, "%s/%s" % (name, pname))


def chunk_check_rows(T, chunk, every=16):
    rows = set(range(0, T, every))
    rows.add(T - 1)
    for c in range(chunk, T, chunk):
        rows.update((c - 1, c))
    return np.array(sorted(rows), np.int64)


@pytest.mark.gpu
def test_long_chunked_prefill_vs_oracle(cuda_device):
    """31,258 tokens in chunks of 4,864 (the last 2,074) through the
    8B-shaped Q4_K layer, issued as the benchmark issues it."""
    t = torch()
    wl = workloads.WORKLOADS["qwen3_8b_q4k_t31258_chunk4864"]
    T, chunk = wl["T"], wl["chunk"]
    assert T - (T // chunk) * chunk == 2074
    X = layer_inputs(wl)
    Xd = {k: dev(v) for k, v in X.items()}
    W = [synth.blocks(qt, out_f, in_f, seed=wl["seed"], tensor=i)
         for i, (_, out_f, in_f, _, qt) in enumerate(wl["projections"])]
    Wd = [dev(w) for w in W]
    Y = [t.full((T, out_f), float("nan"), dtype=t.float32, device="cuda")
         for (_, out_f, _, _, _) in wl["projections"]]
    issue_layer(wl, Wd, Xd, Y, chunk=chunk)
    rows = chunk_check_rows(T, chunk)
    assert rows.size > T // 16
    for i, (pname, out_f, in_f, src, qt) in enumerate(wl["projections"]):
        W32 = oracle.dequant_f32(qt, W[i], out_f, in_f)
        check_rows(Y[i], X[src], W32, rows, "chunked/%s" % pname)
        del W32
    # the same prompt unchunked, and chunked over cached f16 weights: bitwise
    # the chunked fused result, over every element
    for i, (pname, out_f, in_f, src, qt) in enumerate(wl["projections"]):
        if pname not in ("k", "down"):
            continue                      # two projections cover both input widths
        Yu = t.empty_like(Y[i])
        qp.qp_prefill_gemm(qt, Wd[i], out_f, in_f, Xd[src], T, Yu)
        qp.qp_check()
        assert t.equal(Y[i].view(t.int32), Yu.view(t.int32)), pname
        del Yu
        W16 = t.empty((out_f, in_f), dtype=t.float16, device="cuda")
        qp.qp_dequant_f16(qt, Wd[i], out_f, in_f, W16)
        Yh = t.empty_like(Y[i])
        qp.qp_prefill_chunked(qt, None, W16, out_f, in_f, Xd[src], T, Yh, chunk, 1)
        qp.qp_check()
        assert t.equal(Y[i].view(t.int32), Yh.view(t.int32)), pname
        del Yh, W16


def test_chunk_check_rows_cover_every_boundary():
    """(host) The rows the chunked check reads: both sides of every chunk
    boundary, the last row, every 16th row."""
    rows = chunk_check_rows(31258, 4864)
    for c in range(4864, 31258, 4864):
        assert c - 1 in rows and c in rows
    assert 31257 in rows and 0 in rows and 16 in rows
    assert np.all(np.diff(rows) > 0)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["qwen3_8b_q2k_q6k_t8192", "qwen3_8b_q4k_t31258_chunk4864", "qwen3_8b_q5k_t8192"])
@pytest.mark.parametrize("T", [1, 8])
def test_full_size_decode_gemv_every_output_vs_oracle(cuda_device, name, T):
    """The decode GEMV over a whole 8B-shaped layer's weights, issued as the
    benchmark issues it (one grouped launch per run of one block type, here
    for T = 1 and 8 token rows): every element of all seven outputs against
    the fp64 oracle at the workload tolerance."""
    t = torch()
    wl = workloads.WORKLOADS[name]
    dims = workloads.input_dims(wl)
    X = {k: synth.normal_f16((T, dims[k]), seed=wl["seed"], tensor=3000 + i) for i, k in enumerate(dims)}
    Xd = {k: dev(v) for k, v in X.items()}
    W = [synth.blocks(qt, out_f, in_f, seed=wl["seed"], tensor=i)
         for i, (_, out_f, in_f, _, qt) in enumerate(wl["projections"])]
    Wd = [dev(w) for w in W]
    Y = [t.full((T, out_f), float("nan"), dtype=t.float32, device="cuda")
         for (_, out_f, _, _, _) in wl["projections"]]
    for qt, idx in workloads.type_runs(wl["projections"]):
        descs = [(Wd[i], wl["projections"][i][1], wl["projections"][i][2], Xd[wl["projections"][i][3]], Y[i])
                 for i in idx]
        qp.qp_decode_gemv_group(qt, descs, T)
    qp.qp_check()
    rows = np.arange(T, dtype=np.int64)
    for i, (pname, out_f, in_f, src, qt) in enumerate(wl["projections"]):
        W32 = oracle.dequant_f32(qt, W[i], out_f, in_f)
        check_rows(Y[i], X[src], W32, rows, "gemv %s/%s T=%d" % (name, pname, T))
