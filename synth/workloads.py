"""Shapes and seeds of the synthetic workloads (input recipes only).

Layer shapes follow the Qwen3 family: a transformer layer has seven
projections, q/k/v/o in attention and gate/up/down in the MLP.  The q, k, v,
gate and up projections read the same hidden-state input X_h [T x hidden];
o reads its own attention-output input X_o [T x hidden] and down its MLP
input X_f [T x ffn] (there is no attention or MLP between them here, so each
is an independent standard-normal fp16 tensor).  Weights are [out x in].
"""
from . import Q2_K, Q4_K, Q5_K, Q6_K, Q8_0

# (name, out, in, input)
def layer_shapes(hidden, kv, ffn):
    return [("q", hidden, hidden, "h"), ("k", kv, hidden, "h"), ("v", kv, hidden, "h"),
            ("o", hidden, hidden, "o"), ("gate", ffn, hidden, "h"), ("up", ffn, hidden, "h"),
            ("down", hidden, ffn, "f")]


QWEN3_1P7B = dict(hidden=2048, kv=1024, ffn=6144)
QWEN3_8B = dict(hidden=4096, kv=1024, ffn=12288)

WORKLOADS = {
    # Q8_0 256x512 weight, 16 tokens, seed 0
    "q8_0_tiny": dict(seed=0, T=16, projections=[("w", 256, 512, "h", Q8_0)], dims=dict(hidden=512, ffn=512)),
    # Qwen3-1.7B-shaped layer, all Q4_K, 2048 tokens
    "qwen3_1p7b_q4k_t2048": dict(seed=2, T=2048, dims=QWEN3_1P7B,
                                 projections=[p + (Q4_K,) for p in layer_shapes(**QWEN3_1P7B)]),
    # Qwen3-8B-shaped layer, Q2_K everywhere but a Q6_K down projection, 8192 tokens
    "qwen3_8b_q2k_q6k_t8192": dict(seed=3, T=8192, dims=QWEN3_8B,
                                   projections=[p + (Q6_K if p[0] == "down" else Q2_K,)
                                                for p in layer_shapes(**QWEN3_8B)]),
    # Qwen3-8B-shaped layer, all Q4_K, a 31,258-token prompt in chunks of 4,864
    "qwen3_8b_q4k_t31258_chunk4864": dict(seed=4, T=31258, chunk=4864, dims=QWEN3_8B,
                                          projections=[p + (Q4_K,) for p in layer_shapes(**QWEN3_8B)]),
    # Qwen3-8B-shaped layer, all Q5_K, 8192 tokens (the Q5_K row of the next types)
    "qwen3_8b_q5k_t8192": dict(seed=5, T=8192, dims=QWEN3_8B,
                               projections=[p + (Q5_K,) for p in layer_shapes(**QWEN3_8B)]),
}

# Dequant sweep: Q4_K 4096x4096 and 37x1000 (last superblock of each row holds 232 values).
DEQUANT_SWEEP = [("Q4_K", Q4_K, 4096, 4096), ("Q4_K", Q4_K, 37, 1000)]


def type_runs(projections, max_group=8):
    """How a layer is issued: each run of consecutive projections of one
    block type (at most max_group) is one grouped launch.  Returns
    [(type, [projection indices])]."""
    out = []
    for i, p in enumerate(projections):
        qt = p[4]
        if out and out[-1][0] == qt and len(out[-1][1]) < max_group:
            out[-1][1].append(i)
        else:
            out.append((qt, [i]))
    return out


def input_dims(wl):
    d = wl["dims"]
    return {"h": d["hidden"], "o": d["hidden"], "f": d["ffn"]}


def flops(wl, T=None):
    T = wl["T"] if T is None else T
    return sum(2 * T * out * inp for _, out, inp, _, _ in wl["projections"])
