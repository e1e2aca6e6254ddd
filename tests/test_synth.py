"""The seeded generator: deterministic, stream-separated, and drawing the
distributions the workloads state (scales U(1e-3, 1e-2) on the fp16 grid,
uniform packed fields, int8 U[-127, 127], X ~ N(0, 1) on the fp16 grid)."""
import numpy as np

import synth


def test_deterministic_and_separated():
    a = synth.blocks(synth.Q4_K, 16, 512, seed=1, tensor=3)
    b = synth.blocks(synth.Q4_K, 16, 512, seed=1, tensor=3)
    c = synth.blocks(synth.Q4_K, 16, 512, seed=1, tensor=4)
    d = synth.blocks(synth.Q4_K, 16, 512, seed=2, tensor=3)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)
    x = synth.normal_f16((64, 64), seed=0)
    assert np.array_equal(x.view(np.uint16), synth.normal_f16((64, 64), seed=0).view(np.uint16))


def test_prefix_stable():
    """Block b depends only on (seed, tensor, b): a bigger tensor starts with
    the same blocks."""
    a = synth.blocks(synth.Q6_K, 4, 256, seed=9).ravel()
    b = synth.blocks(synth.Q6_K, 8, 256, seed=9).ravel()
    assert np.array_equal(a, b[:a.size])


def test_scale_fields_in_range():
    for qtype, off in ((synth.Q8_0, [0]), (synth.Q4_K, [0, 2]), (synth.Q2_K, [80, 82]), (synth.Q6_K, [208])):
        w = synth.blocks(qtype, 64, 1024, seed=5, tensor=qtype)
        bb = synth.BLOCK[qtype][1]
        blk = w.reshape(-1, bb)
        for o in off:
            d = blk[:, o:o + 2].copy().view(np.float16).astype(np.float64).ravel()
            assert d.min() >= 1e-3 * (1 - 2 ** -11) and d.max() <= 1e-2 * (1 + 2 ** -11)
            assert 4.5e-3 < d.mean() < 6.5e-3


def test_int8_fields_symmetric_without_minus_128():
    w = synth.blocks(synth.Q8_0, 256, 1024, seed=6).reshape(-1, 34)
    q = w[:, 2:].view(np.int8).ravel()
    assert q.min() == -127 and q.max() == 127 and abs(q.mean()) < 1.0
    s = synth.blocks(synth.Q6_K, 256, 1024, seed=6).reshape(-1, 210)[:, 192:208].view(np.int8).ravel()
    assert s.min() >= -127 and s.max() <= 127


def test_uniform_packed_fields():
    qs = synth.blocks(synth.Q4_K, 256, 1024, seed=7).reshape(-1, 144)[:, 16:].ravel()
    counts = np.bincount(np.concatenate([qs & 15, qs >> 4]), minlength=16)
    assert counts.min() > 0.95 * counts.mean() and counts.max() < 1.05 * counts.mean()


def test_normal_moments():
    x = synth.normal_f16((1 << 20,), seed=3).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1) < 5e-3
    assert np.all(np.isfinite(x))


def test_anybits_blocks_cover_every_field_pattern():
    """blocks_anybits: every quant/scale byte value occurs (int8 -128 included),
    while d and dmin are drawn as for blocks (finite, U(1e-3, 1e-2) on the fp16
    grid)."""
    d_offsets = {synth.Q8_0: [0], synth.Q4_K: [0, 2], synth.Q5_K: [0, 2], synth.Q2_K: [80, 82],
                 synth.Q6_K: [208]}
    for qtype, offs in d_offsets.items():
        bb = synth.BLOCK[qtype][1]
        w = synth.blocks_anybits(qtype, 64, 2048, seed=11, tensor=qtype).reshape(-1, bb)
        field = np.ones(bb, bool)
        for o in offs:
            field[o:o + 2] = False
            d = w[:, o:o + 2].copy().view(np.float16).astype(np.float64).ravel()
            assert d.min() >= 1e-3 * (1 - 2 ** -11) and d.max() <= 1e-2 * (1 + 2 ** -11)
        counts = np.bincount(w[:, field].ravel(), minlength=256)
        assert counts.min() > 0.5 * counts.mean(), qtype
    s = synth.blocks_anybits(synth.Q6_K, 64, 2048, seed=11, tensor=14).reshape(-1, 210)[:, 192:208]
    assert (s.view(np.int8) == -128).any()
    f = synth.blocks_anybits(synth.F16, 8, 64, seed=1, tensor=1)
    assert np.array_equal(f, synth.blocks(synth.F16, 8, 64, seed=1, tensor=1))
