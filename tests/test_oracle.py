"""Pins of the CPU oracle against things other than itself.

- hand-worked blocks (tests/golden/), values worked out by hand;
- fp16 conversions against numpy's IEEE conversions (exhaustive / ties);
- the value formulas in closed form, evaluated exactly in fp64 on fields
  packed by an independent test-side packer;
- structure of every format by bit flips: each quant bit moves exactly one
  value by the bit's weight, each scale bit moves exactly one aligned
  sub-block, so a dropped, doubled or mis-shifted field cannot pass;
- brute-force requantize / dequantize round trips on tiny tensors;
- partial last blocks and the row stride;
- the fp64 GEMM against numpy's fp64 matmul and a hand-summed case.
"""
import itertools

import numpy as np
import pytest

import oracle
import synth
from golden_blocks import fixtures, load

Q8_0, Q2_K, Q4_K, Q5_K, Q6_K = oracle.Q8_0, oracle.Q2_K, oracle.Q4_K, oracle.Q5_K, oracle.Q6_K
F16 = oracle.F16
ALL = [Q8_0, Q2_K, Q4_K, Q5_K, Q6_K]


def f16bits(x):
    return np.array([x], np.float16).view(np.uint16)[0]


# --------------------------------------------------------------- golden ---

@pytest.mark.parametrize("path", fixtures(), ids=lambda p: p.rsplit("/", 1)[-1])
def test_golden_block(path):
    qtype, block, expected = load(path)
    got = np.array([oracle.decode_value(qtype, block, v) for v in range(expected.size)])
    np.testing.assert_array_equal(got, expected)
    # the row form decodes the same block the same way
    row = oracle.dequant_f32(qtype, block, 1, expected.size)[0]
    np.testing.assert_array_equal(row.astype(np.float64), expected)


# ----------------------------------------------------------------- fp16 ---

def test_f16_to_f32_exhaustive_vs_numpy():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_f16_ties_and_boundaries_vs_numpy():
    # every finite fp16 value, and every midpoint between neighbours (ties),
    # and points a hair either side of each midpoint
    h = np.arange(0, 0x7c00, dtype=np.uint32).astype(np.uint16)
    v = h.view(np.float16).astype(np.float64)
    mids = (v[:-1] + v[1:]) / 2
    cands = [v, mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf),
             np.array([65504.0, 65519.0, 65520.0, 65536.0, 1e9, 2.0 ** -25, 2.0 ** -26, 2.0 ** -24 * 1.5])]
    f = np.concatenate(cands).astype(np.float32)
    f = np.concatenate([f, -f, np.array([np.inf, -np.inf, 0.0, -0.0], np.float32)])
    got = oracle.f32_to_f16(f)
    ref = f.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_f32_to_f16_random_bits_vs_numpy():
    bits = synth.random_bytes(4 * 2_000_000, seed=7).view(np.uint32)
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    got = oracle.f32_to_f16(f)
    ref = f.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_f32_to_f16_nan_stays_nan():
    got = oracle.f32_to_f16(np.array([np.nan, -np.nan], np.float32))
    assert np.all(np.isnan(got.view(np.float16)))


# ------------------------------------------- independent test-side packers ---
# Written from the layout description (GGUF reading), in the opposite direction
# of the oracle's decoder: fields in, bytes out.

def pack_q8_0(d, q):
    b = np.zeros(34, np.uint8)
    b[0:2] = np.array([d], np.float16).view(np.uint8)
    b[2:34] = np.asarray(q, np.int8).view(np.uint8)
    return b


def pack_q4_k(d, dmin, sc, m, q):
    b = np.zeros(144, np.uint8)
    b[0:2] = np.array([d], np.float16).view(np.uint8)
    b[2:4] = np.array([dmin], np.float16).view(np.uint8)
    s = np.zeros(12, np.int64)
    for j in range(4):
        s[j] = sc[j] | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = m[j] | ((m[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    b[4:16] = s
    qs = np.zeros(128, np.int64)
    for v in range(256):
        g, l = v // 64, v % 32
        qs[32 * g + l] |= q[v] if v % 64 < 32 else q[v] << 4
    b[16:144] = qs
    return b


def pack_q5_k(d, dmin, sc, m, q):
    """Q4_K's fields with 5-bit q: the low four bits where Q4_K keeps q, the
    fifth bit of value v in bit v//32 of qh[v % 32] (qh sits before qs)."""
    b4 = pack_q4_k(d, dmin, sc, m, np.asarray(q) & 15)
    b = np.zeros(176, np.uint8)
    b[0:16] = b4[0:16]
    qh = np.zeros(32, np.int64)
    for v in range(256):
        qh[v % 32] |= (int(q[v]) >> 4) << (v // 32)
    b[16:48] = qh
    b[48:176] = b4[16:144]
    return b


def pack_q2_k(d, dmin, sc, m, q):
    b = np.zeros(84, np.uint8)
    b[0:16] = np.asarray(sc) | (np.asarray(m) << 4)
    qs = np.zeros(64, np.int64)
    for v in range(256):
        n, j, l = v // 128, (v % 128) // 32, v % 32
        qs[32 * n + l] |= q[v] << (2 * j)
    b[16:80] = qs
    b[80:82] = np.array([d], np.float16).view(np.uint8)
    b[82:84] = np.array([dmin], np.float16).view(np.uint8)
    return b


def pack_q6_k(d, s, q):
    b = np.zeros(210, np.uint8)
    ql = np.zeros(128, np.int64)
    qh = np.zeros(64, np.int64)
    for v in range(256):
        n, j, l = v // 128, (v % 128) // 32, v % 32
        lo, hi = q[v] & 15, q[v] >> 4
        idx = 64 * n + l + 32 * (j & 1)
        ql[idx] |= lo if j < 2 else lo << 4
        qh[32 * n + l] |= hi << (2 * j)
    b[0:128] = ql
    b[128:192] = qh
    b[192:208] = np.asarray(s, np.int8).view(np.uint8)
    b[208:210] = np.array([d], np.float16).view(np.uint8)
    return b


def exact_f32(x):
    """fp64 value (exact here) rounded once to f32."""
    return np.float32(x)


def rand_fields(rng, qtype):
    d = float(np.float16(rng.uniform(1e-3, 1e-2)))
    dmin = float(np.float16(rng.uniform(1e-3, 1e-2)))
    if qtype == Q8_0:
        return d, None, None, None, rng.integers(-127, 128, 32)
    if qtype == Q4_K:
        return d, dmin, rng.integers(0, 64, 8), rng.integers(0, 64, 8), rng.integers(0, 16, 256)
    if qtype == Q5_K:
        return d, dmin, rng.integers(0, 64, 8), rng.integers(0, 64, 8), rng.integers(0, 32, 256)
    if qtype == Q2_K:
        return d, dmin, rng.integers(0, 16, 16), rng.integers(0, 16, 16), rng.integers(0, 4, 256)
    return d, None, rng.integers(-127, 128, 16), None, rng.integers(0, 64, 256)


def closed_form(qtype, d, dmin, sc, m, q):
    """Value formulas of the workload definition, in exact fp64."""
    if qtype == Q8_0:
        return [d * q[v] for v in range(32)]
    if qtype in (Q4_K, Q5_K):
        return [d * sc[v // 32] * q[v] - dmin * m[v // 32] for v in range(256)]
    if qtype == Q2_K:
        return [d * sc[v // 16] * q[v] - dmin * m[v // 16] for v in range(256)]
    return [d * sc[v // 16] * (q[v] - 32) for v in range(256)]


def pack(qtype, d, dmin, sc, m, q):
    if qtype == Q8_0:
        return pack_q8_0(d, q)
    if qtype == Q4_K:
        return pack_q4_k(d, dmin, sc, m, q)
    if qtype == Q5_K:
        return pack_q5_k(d, dmin, sc, m, q)
    if qtype == Q2_K:
        return pack_q2_k(d, dmin, sc, m, q)
    return pack_q6_k(d, sc, q)


@pytest.mark.parametrize("qtype", ALL)
def test_closed_form_on_packed_fields(qtype):
    rng = np.random.default_rng(qtype)
    qk = oracle.BLOCK[qtype][0]
    for _ in range(40):
        f = rand_fields(rng, qtype)
        block = pack(qtype, *f)
        got = oracle.dequant_f32(qtype, block, 1, qk)[0]
        want = np.array([exact_f32(x) for x in closed_form(qtype, *f)], np.float32)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_q4_k_every_scale_min_pair_at_every_position():
    """All 64x64 (sc, m) pairs at each of the 8 packed positions."""
    d, dmin = 2.0 ** -6, 2.0 ** -7
    q = np.full(256, 15)
    sc_all, m_all = np.meshgrid(np.arange(64), np.arange(64))
    for pos in range(8):
        for sc_v, m_v in zip(sc_all.ravel()[::7], m_all.ravel()[::7]):
            sc = np.full(8, 5)
            m = np.full(8, 9)
            sc[pos], m[pos] = sc_v, m_v
            got = oracle.dequant_f32(Q4_K, pack_q4_k(d, dmin, sc, m, q), 1, 256)[0]
            want = np.float32(d * sc_v * 15 - dmin * m_v)
            assert np.all(got[32 * pos:32 * pos + 32] == want)
        # the exhaustive pass over all pairs at this position
        sc = np.full(8, 5)
        m = np.full(8, 9)
        for sc_v in range(64):
            for m_v in range(64):
                sc[pos], m[pos] = sc_v, m_v
                b = pack_q4_k(d, dmin, sc, m, q)
                v0 = oracle.decode_value(Q4_K, b, 32 * pos)
                assert v0 == np.float32(d * sc_v * 15 - dmin * m_v)


def test_nibble_and_crumb_extraction_all_bytes():
    """Every byte value in every qs position decodes to the right nibble / crumb."""
    d, dmin = 1.0, 0.0
    for byte in range(256):
        b = pack_q4_k(d, dmin, np.ones(8, int), np.zeros(8, int), np.zeros(256, int))
        b[16:144] = byte
        vals = oracle.dequant_f32(Q4_K, b, 1, 256)[0]
        for v in range(256):
            assert vals[v] == (byte & 15 if v % 64 < 32 else byte >> 4)
        b = pack_q2_k(d, dmin, np.ones(16, int), np.zeros(16, int), np.zeros(256, int))
        b[16:80] = byte
        vals = oracle.dequant_f32(Q2_K, b, 1, 256)[0]
        for v in range(256):
            assert vals[v] == (byte >> (2 * ((v % 128) // 32))) & 3


def test_q5_k_high_bit_extraction_all_bytes():
    """Every qh byte value at every qh position: value v gets bit v//32 of
    qh[v % 32] as its fifth bit (q = 16 * that bit with the nibbles zero)."""
    b = pack_q5_k(1.0, 0.0, np.ones(8, int), np.zeros(8, int), np.zeros(256, int))
    for byte in range(256):
        b[16:48] = byte
        vals = oracle.dequant_f32(Q5_K, b, 1, 256)[0]
        for v in range(256):
            assert vals[v] == 16 * ((byte >> (v // 32)) & 1)
    for l in range(32):                      # one position at a time
        b[16:48] = 0
        b[16 + l] = 0xff
        vals = oracle.dequant_f32(Q5_K, b, 1, 256)[0]
        assert np.array_equal(np.nonzero(vals)[0], np.arange(l, 256, 32))


def test_q6_k_all_low_high_combinations():
    d = 1.0
    for lo, hi in itertools.product(range(16), range(4)):
        q = np.full(256, lo | (hi << 4))
        b = pack_q6_k(d, np.ones(16, int), q)
        vals = oracle.dequant_f32(Q6_K, b, 1, 256)[0]
        assert np.all(vals == (lo | (hi << 4)) - 32)


# ------------------------------------------------------------ bit flips ---
# Reading-independent structure checks.

QREGION = {Q8_0: (2, 34), Q4_K: (16, 144), Q5_K: (16, 176), Q2_K: (16, 80), Q6_K: (0, 192)}
SREGION = {Q4_K: (4, 16), Q5_K: (4, 16), Q2_K: (0, 16), Q6_K: (192, 208)}
DOFF = {Q8_0: 0, Q4_K: 0, Q5_K: 0, Q2_K: 80, Q6_K: 208}
QBITS = {Q8_0: 8, Q4_K: 4, Q5_K: 5, Q2_K: 2, Q6_K: 6}
SUB = {Q4_K: 32, Q5_K: 32, Q2_K: 16, Q6_K: 16}


def base_block(qtype, q_ones):
    """d = 2^-6 (dmin = 2^-7); every scale field at a nonzero value; the quant
    region all zero, or all ones when q_ones."""
    bb = oracle.BLOCK[qtype][1]
    b = np.zeros(bb, np.uint8)
    b[DOFF[qtype]:DOFF[qtype] + 2] = np.array([2.0 ** -6], np.float16).view(np.uint8)
    if qtype in (Q4_K, Q5_K, Q2_K):
        off = 82 if qtype == Q2_K else 2
        b[off:off + 2] = np.array([2.0 ** -7], np.float16).view(np.uint8)
    lo, hi = QREGION[qtype]
    if q_ones:
        b[lo:hi] = 0xff
    return b


@pytest.mark.parametrize("qtype", ALL)
def test_every_quant_bit_moves_exactly_one_value(qtype):
    qk = oracle.BLOCK[qtype][0]
    b0 = base_block(qtype, q_ones=False)
    if qtype in SREGION:
        lo, hi = SREGION[qtype]
        b0[lo:hi] = 0xff if qtype != Q6_K else 0x01
    y0 = oracle.dequant_f32(qtype, b0, 1, qk)[0].astype(np.float64)
    hits = {v: [] for v in range(qk)}
    lo, hi = QREGION[qtype]
    for byte in range(lo, hi):
        for bit in range(8):
            b = b0.copy()
            b[byte] ^= 1 << bit
            y = oracle.dequant_f32(qtype, b, 1, qk)[0].astype(np.float64)
            moved = np.nonzero(y != y0)[0]
            assert moved.size == 1, (byte, bit, moved)
            v = int(moved[0])
            hits[v].append(y[v] - y0[v])
    for v in range(qk):
        steps = sorted(hits[v])
        assert len(steps) == QBITS[qtype], (v, steps)
        # the steps are the bit weights of one n-bit field times one scale
        unit = min(abs(s) for s in steps)
        weights = sorted(round(s / unit) for s in steps)
        if qtype == Q8_0:
            assert weights == [-128, 1, 2, 4, 8, 16, 32, 64]
        else:
            assert weights == [2 ** k for k in range(QBITS[qtype])]


@pytest.mark.parametrize("qtype", [Q4_K, Q5_K, Q2_K, Q6_K])
def test_every_scale_bit_moves_one_aligned_subblock(qtype):
    qk = oracle.BLOCK[qtype][0]
    b0 = base_block(qtype, q_ones=True)
    y0 = oracle.dequant_f32(qtype, b0, 1, qk)[0].astype(np.float64)
    sub = SUB[qtype]
    per_sub = {s: [] for s in range(qk // sub)}
    lo, hi = SREGION[qtype]
    for byte in range(lo, hi):
        for bit in range(8):
            b = b0.copy()
            b[byte] ^= 1 << bit
            y = oracle.dequant_f32(qtype, b, 1, qk)[0].astype(np.float64)
            moved = np.nonzero(y != y0)[0]
            assert moved.size == sub, (byte, bit, moved)
            s = moved[0] // sub
            assert moved[0] == s * sub and np.all(moved == np.arange(s * sub, s * sub + sub))
            delta = y[moved] - y0[moved]
            assert np.all(delta == delta[0])        # q is constant, so one step
            per_sub[s].append(delta[0])
    d, dmin = 2.0 ** -6, 2.0 ** -7
    for s, deltas in per_sub.items():
        if qtype in (Q4_K, Q5_K):   # 6-bit sc (step d*qmax*2^k) and 6-bit m (step -dmin*2^k)
            qmax = 15 if qtype == Q4_K else 31
            sc_w = sorted(round(x / (d * qmax)) for x in deltas if x > 0)
            m_w = sorted(round(-x / dmin) for x in deltas if x < 0)
            assert sc_w == [1, 2, 4, 8, 16, 32] and m_w == [1, 2, 4, 8, 16, 32], (s, deltas)
        elif qtype == Q2_K:    # 4-bit sc (d*3*2^k) and 4-bit m (-dmin*2^k)
            sc_w = sorted(round(x / (d * 3)) for x in deltas if x > 0)
            m_w = sorted(round(-x / dmin) for x in deltas if x < 0)
            assert sc_w == [1, 2, 4, 8] and m_w == [1, 2, 4, 8], (s, deltas)
        else:                  # int8 scale, q - 32 = 31
            w = sorted(round(x / (d * 31)) for x in deltas)
            assert w == [-128, 1, 2, 4, 8, 16, 32, 64], (s, deltas)


# ----------------------------------------------------------- round trip ---

def requant_search(qtype, d, dmin, y):
    """Brute force: for each sub-block find fields whose decoded f32 values
    reproduce y exactly (f32 arithmetic, each operation rounded)."""
    f = np.float32
    d, dmin = f(d), f(dmin)
    if qtype in (Q4_K, Q5_K):
        nsub, sub, scr, qr = 8, 32, 64, 16 if qtype == Q4_K else 32
    else:
        nsub, sub, scr, qr = 16, 16, 16, 4
    sc_out, m_out, q_out = [], [], np.zeros(256, np.int64)
    for s in range(nsub):
        ys = y[s * sub:(s + 1) * sub]
        found = False
        for sc in range(scr):
            dl = f(d * f(sc))
            for m in range(scr):
                ml = f(dmin * f(m))
                table = np.array([f(f(dl * f(q)) - ml) for q in range(qr)], np.float32)
                idx = [np.nonzero(table.view(np.uint32) == yy.view(np.uint32))[0] for yy in ys]
                if all(i.size for i in idx):
                    sc_out.append(sc)
                    m_out.append(m)
                    q_out[s * sub:(s + 1) * sub] = [i[0] for i in idx]
                    found = True
                    break
            if found:
                break
        assert found, s
    return sc_out, m_out, q_out


@pytest.mark.parametrize("qtype", [Q4_K, Q5_K, Q2_K])
def test_requant_round_trip(qtype):
    w = synth.blocks(qtype, 1, 256, seed=11, tensor=qtype)
    y = oracle.dequant_f32(qtype, w, 1, 256)[0]
    dof = 80 if qtype == Q2_K else 0
    d = float(w[0, dof:dof + 2].view(np.float16)[0])
    dmin = float(w[0, dof + 2:dof + 4].view(np.float16)[0])
    sc, m, q = requant_search(qtype, d, dmin, y)
    packer = {Q4_K: pack_q4_k, Q5_K: pack_q5_k, Q2_K: pack_q2_k}[qtype]
    b2 = packer(d, dmin, np.array(sc), np.array(m), q)
    y2 = oracle.dequant_f32(qtype, b2, 1, 256)[0]
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


def test_q8_0_and_q6_k_round_trip():
    for qtype in (Q8_0, Q6_K):
        qk = oracle.BLOCK[qtype][0]
        w = synth.blocks(qtype, 1, qk, seed=12, tensor=qtype)
        y = oracle.dequant_f32(qtype, w, 1, qk)[0]
        if qtype == Q8_0:
            d = np.float32(w[0, 0:2].view(np.float16)[0])
            q = [next(k for k in range(-127, 128) if np.float32(d * np.float32(k)) == yy) for yy in y]
            b2 = pack_q8_0(float(d), q)
        else:
            d = np.float32(w[0, 208:210].view(np.float16)[0])
            s = w[0, 192:208].view(np.int8).astype(np.int64)
            q = [next(k for k in range(64)
                      if np.float32(np.float32(d * np.float32(s[v // 16])) * np.float32(k - 32)) == y[v])
                 for v in range(256)]
            b2 = pack_q6_k(float(d), s, np.array(q))
        y2 = oracle.dequant_f32(qtype, b2, 1, qk)[0]
        assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


# ------------------------------------------------ rows, tails, f16 copy ---

@pytest.mark.parametrize("qtype", ALL)
def test_partial_last_block_and_row_stride(qtype):
    qk, bb = oracle.BLOCK[qtype]
    rows, nb = 5, 4
    w = synth.blocks(qtype, rows, nb * qk, seed=3, tensor=qtype)
    full = oracle.dequant_f32(qtype, w, rows, nb * qk)
    for cols in (nb * qk - 1, (nb - 1) * qk + 1, (nb - 1) * qk + qk // 2 + 3):
        part = oracle.dequant_f32(qtype, w, rows, cols)
        assert part.shape == (rows, cols)
        assert np.array_equal(part, full[:, :cols])


def test_partial_block_config_shape():
    """37 x 1000 Q4_K: 4 superblocks per row, the last holding 232 values."""
    w = synth.blocks(Q4_K, 37, 1000, seed=2, tensor=1)
    assert w.shape == (37, 4 * 144)
    y = oracle.dequant_f32(Q4_K, w, 37, 1000)
    full = oracle.dequant_f32(Q4_K, w, 37, 1024)
    assert np.array_equal(y, full[:, :1000])


@pytest.mark.parametrize("qtype", ALL)
def test_f16_copy_is_rounded_f32_result(qtype):
    qk = oracle.BLOCK[qtype][0]
    w = synth.blocks(qtype, 8, 3 * qk, seed=4, tensor=qtype)
    y32 = oracle.dequant_f32(qtype, w, 8, 3 * qk)
    y16 = oracle.dequant_f16(qtype, w, 8, 3 * qk)
    assert np.array_equal(y16, y32.astype(np.float16).view(np.uint16))


def test_nan_and_inf_scales_propagate():
    b = pack_q8_0(1.0, np.arange(32) - 16)
    b[0:2] = np.array([f16bits(np.inf)]).view(np.uint8)
    y = oracle.dequant_f32(Q8_0, b, 1, 32)[0]
    assert np.isnan(y[16])                      # inf * 0
    assert np.all(np.isinf(y[np.arange(32) != 16]))
    b[0:2] = np.array([0x7e00], np.uint16).view(np.uint8)
    assert np.all(np.isnan(oracle.dequant_f32(Q8_0, b, 1, 32)))


def test_bad_type_rejected():
    with pytest.raises(KeyError):
        oracle.dequant_f32(11, np.zeros(16, np.uint8), 1, 16)
    assert oracle.lib().qpo_dequant_f32(11, None, 1, 1, None) == -1


def test_f16_weights_decode_to_their_value_for_every_bit_pattern():
    """F16 "blocks" are single fp16 weights: the f32 dequant is the exact
    widening (numpy's IEEE conversion), the f16 dequant gives the same bits
    back (NaNs stay NaN)."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    y = oracle.dequant_f32(F16, h.view(np.uint8), 1, 65536)[0]
    want = h.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(y), nan)
    assert np.array_equal(y[~nan].view(np.uint32), want[~nan].view(np.uint32))
    y16 = oracle.dequant_f16(F16, h.view(np.uint8), 1, 65536)[0]
    assert np.array_equal(y16[~nan], h[~nan])
    assert np.all(np.isnan(y16[nan].view(np.float16)))


# ----------------------------------------------------------------- GEMM ---

def test_gemm_hand_summed():
    X = np.array([[1, 2, 0.5, -1], [0, 0, 0, 1]], np.float16)
    W = np.array([[1, 1, 1, 1], [2, 0, -1, 0.25], [0, 0, 0, 0]], np.float32)
    Y, A = oracle.gemm_f64(X, W)
    assert np.array_equal(Y, [[2.5, 1.25, 0.0], [1.0, 0.25, 0.0]])
    assert np.array_equal(A, [[4.5, 2.75, 0.0], [1.0, 0.25, 0.0]])


def test_gemm_vs_numpy_fp64_matmul():
    X = synth.normal_f16((37, 512), seed=5)
    w = synth.blocks(Q4_K, 24, 512, seed=5, tensor=1)
    W = oracle.dequant_f32(Q4_K, w, 24, 512)
    Y, A = oracle.gemm_f64(X, W)
    Xd = X.astype(np.float64)
    Wd = W.astype(np.float64)
    np.testing.assert_allclose(Y, Xd @ Wd.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(A, np.abs(Xd) @ np.abs(Wd).T, rtol=1e-12, atol=1e-12)
    assert np.all(A >= np.abs(Y))


def test_gemm_row_subset_matches_full():
    X = synth.normal_f16((20, 256), seed=6)
    W = oracle.dequant_f32(Q2_K, synth.blocks(Q2_K, 16, 256, seed=6), 16, 256)
    Y, A = oracle.gemm_f64(X, W)
    rows = np.array([19, 0, 7, 7])
    Ys, As = oracle.gemm_f64(X, W, rows)
    assert np.array_equal(Ys, Y[rows]) and np.array_equal(As, A[rows])


def test_gemm_one_hot_rows_select_weight_columns():
    W = oracle.dequant_f32(Q6_K, synth.blocks(Q6_K, 8, 256, seed=8), 8, 256)
    X = np.zeros((4, 256), np.float16)
    ks = [0, 17, 128, 255]
    for t, k in enumerate(ks):
        X[t, k] = 1
    Y, _ = oracle.gemm_f64(X, W)
    for t, k in enumerate(ks):
        assert np.array_equal(Y[t], W[:, k].astype(np.float64))
