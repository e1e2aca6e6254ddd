"""GPU parity of qp_dequant_f32 / qp_dequant_f16 against the CPU oracle: bit
for bit, on NaN-guarded outputs ("Qwen3.5 batched prefill has no f32 dequant
for IQ2_XXS, IQ3_S, IQ3_XXS, Q2_K", §Acceptance: bit-exact, partial last
blocks, NaN-prefilled scratch checked for out-of-bounds writes)."""
import numpy as np
import pytest

import block_quantized_weight_qp_gb300 as qp
import oracle
import synth
from golden_blocks import fixtures, load
from qp_testutil import dev, guard_intact, guarded

pytestmark = pytest.mark.gpu

TYPES = {"Q8_0": qp.Q8_0, "Q2_K": qp.Q2_K, "Q4_K": qp.Q4_K, "Q5_K": qp.Q5_K, "Q6_K": qp.Q6_K, "F16": qp.F16}

SHAPES = [
    ("Q8_0", 256, 512),        # the Q8_0 tiny weight
    ("Q4_K", 4096, 4096),      # the Q4_K sweep, full size
    ("Q4_K", 37, 1000),        # last superblock of each row holds 232 values
    ("Q2_K", 1024, 4096),
    ("Q2_K", 33, 700),
    ("Q6_K", 512, 12288),
    ("Q6_K", 29, 1100),
    ("Q8_0", 31, 1000),        # 32 blocks per row, the last holding 8 values
    ("Q8_0", 7, 33),
    ("Q4_K", 1, 1),
    ("Q2_K", 3, 255),
    ("Q6_K", 5, 256),
    ("Q4_K", 9, 257),
    ("Q8_0", 1, 31),
    ("Q4_K", 3, 4),            # f32 rows 16-byte aligned, f16 rows not
    ("Q6_K", 2, 6),
    ("Q5_K", 1024, 4096),
    ("Q5_K", 37, 1000),
    ("Q5_K", 3, 255),
    ("F16", 256, 512),
    ("F16", 7, 33),            # 231 values: a last partial group of 8
    ("F16", 1, 1),
    ("F16", 3, 1000),
]


def run(qtype, blocks, rows, cols, f16):
    import torch
    d = dev(blocks)
    n = rows * cols
    buf, out, g = guarded(n, torch.float16 if f16 else torch.float32, cols)
    (qp.qp_dequant_f16 if f16 else qp.qp_dequant_f32)(qtype, d, rows, cols, out)
    qp.qp_check()
    assert guard_intact(buf, g, n), "write outside the output"
    return out.cpu().numpy().reshape(rows, cols)


@pytest.mark.parametrize("name,rows,cols", SHAPES, ids=lambda x: str(x))
@pytest.mark.parametrize("f16", [False, True], ids=["f32", "f16"])
def test_dequant_bit_exact(cuda_device, name, rows, cols, f16):
    qtype = TYPES[name]
    w = synth.blocks(qtype, rows, cols, seed=rows * 7 + cols, tensor=qtype)
    got = run(qtype, w, rows, cols, f16)
    if f16:
        want = oracle.dequant_f16(qtype, w, rows, cols)
        assert np.array_equal(got.view(np.uint16), want)
    else:
        want = oracle.dequant_f32(qtype, w, rows, cols)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("path", fixtures(), ids=lambda p: p.rsplit("/", 1)[-1])
def test_dequant_golden_blocks(cuda_device, path):
    qtype, block, expected = load(path)
    qk = expected.size
    rows = 3
    blocks = np.tile(block, rows)
    got = run(qtype, blocks, rows, qk, f16=False)
    assert np.array_equal(got.astype(np.float64), np.tile(expected, (rows, 1)))


def test_dequant_random_bytes_including_specials(cuda_device):
    """Uniform random block bytes: the fp16 scales then include subnormals,
    infinities and NaNs; non-NaN values must match bit for bit and NaNs must
    sit in the same places."""
    for name, qtype in TYPES.items():
        qk, bb = oracle.BLOCK[qtype]
        rows, cols = 64, 8 * qk - 3
        nb = -(-cols // qk)
        w = synth.random_bytes(rows * nb * bb, seed=99, tensor=qtype).reshape(rows, nb * bb)
        for f16 in (False, True):
            got = run(qtype, w, rows, cols, f16)
            want = (oracle.dequant_f16 if f16 else oracle.dequant_f32)(qtype, w, rows, cols)
            gv = got.view(np.uint16 if f16 else np.uint32)
            gnan = np.isnan(got)
            wnan = np.isnan(want.view(np.float16) if f16 else want)
            assert np.array_equal(gnan, wnan), name
            assert np.array_equal(gv[~gnan], want.view(gv.dtype)[~wnan]), name
