"""qp_plan_prefill: the fit rule of "QK-norm models take the FP16 batched
prefill when it fits" (§What changes: weights + FP16 cache + KV + prefill
reserve against free VRAM, from the projection tensors' own bytes), checked
at its boundaries.  Host only, no GPU."""
import pytest

import block_quantized_weight_qp_gb300 as qp

# two projections: Q4_K 512 x 1024 and Q2_K 256 x 2048
SHAPES = [(qp.Q4_K, 512, 1024), (qp.Q2_K, 256, 2048)]
W = 512 * 4 * 144 + 256 * 8 * 84            # quantized bytes, from the block sizes
CACHE = (512 * 1024 + 256 * 2048) * 2       # f16 copies
ACT = (2 * 1024 + 4 * 512) + (2 * 2048 + 4 * 256)
KV, RES = 1000, 24


def plan(free, T=10000, max_chunk=0, shapes=SHAPES):
    return qp.qp_plan_prefill(shapes, T, free, kv_bytes=KV, reserve_bytes=RES, max_chunk=max_chunk)


def test_byte_counts_come_from_the_tensors():
    p = plan(10 ** 12)
    assert (p["weight_bytes"], p["f16_cache_bytes"], p["act_bytes_per_row"]) == (W, CACHE, ACT)


def test_cached_mode_when_everything_fits_and_chunk_is_tile_rounded():
    base = W + CACHE + KV + RES
    p = plan(base + 1000 * ACT + ACT - 1)       # room for 1000.99 rows
    assert p["mode"] == 1 and p["chunk"] == 768  # rounded down to a multiple of 256
    assert p["total_bytes"] == base + 768 * ACT
    p = plan(base + 256 * ACT)                  # exactly 256 rows
    assert p["mode"] == 1 and p["chunk"] == 256
    p = plan(base + 256 * ACT - 1)              # one byte short of 256 rows: 255, not rounded
    assert p["mode"] == 1 and p["chunk"] == 255


def test_fused_mode_when_the_f16_cache_does_not_fit():
    base = W + KV + RES
    p = plan(base + CACHE)                      # the cache fits, but no row beside it
    assert p["mode"] == 0 and p["total_bytes"] == base + p["chunk"] * ACT
    p = plan(base + 3 * ACT)
    assert p["mode"] == 0 and p["chunk"] == 3


def test_does_not_fit():
    p = plan(W + KV + RES + ACT - 1)
    assert p["mode"] == -1 and p["chunk"] == 0 and p["total_bytes"] == 0


def test_prompt_length_and_cap_bound_the_chunk():
    assert plan(10 ** 12, T=100)["chunk"] == 100
    assert plan(10 ** 12, T=10000, max_chunk=4864)["chunk"] == 4864
    assert plan(10 ** 12, T=10000, max_chunk=1000)["chunk"] == 768
    assert plan(10 ** 12, T=31258)["chunk"] == 31258 // 256 * 256


def test_f16_weights_are_their_own_cache():
    p = qp.qp_plan_prefill([(qp.F16, 128, 256)], 512, 10 ** 9)
    assert p["weight_bytes"] == 128 * 256 * 2 and p["f16_cache_bytes"] == 0 and p["mode"] == 1


@pytest.mark.parametrize("args", [
    dict(shapes=[], T=1, free=1), dict(shapes=SHAPES, T=0, free=1), dict(shapes=SHAPES, T=1, free=-1),
    dict(shapes=[(qp.Q4_K, 0, 256)], T=1, free=1),
])
def test_invalid_arguments(args):
    with pytest.raises(qp.QPError) as e:
        qp.qp_plan_prefill(args["shapes"], args["T"], args["free"])
    assert e.value.status == qp.QP_ERR_INVALID_PARAMETER


def test_unsupported_type():
    with pytest.raises(qp.QPError) as e:
        qp.qp_plan_prefill([(11, 256, 256)], 1, 10 ** 9)
    assert e.value.status == qp.QP_ERR_UNSUPPORTED_TYPE
