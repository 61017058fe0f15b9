"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each pin takes the oracle module and raises AssertionError on a mismatch.  The
pins are run directly by tests/test_oracle_pins.py and, against deliberately
broken builds of the oracle, by tests/test_oracle_mutants.py (each planted
mistake must make at least one pin fail).

What each pin rests on:
  * the E2M1 code table and the range facts printed on the page "Gemma 4 NVFP4
    MoE 空输出" (§NVFP4), transcribed into tests/golden/;
  * the rounding rule stated there (nearest, ties to even, saturating),
    restated here as decision boundaries rather than as a nearest-value search;
  * the OCP E4M3FN definition, restated here with frexp, and PyTorch's
    float8_e4m3fn conversion (a library routine) inside the finite range;
  * hand-worked blocks whose codes follow from the code table alone;
  * exact rational arithmetic (fractions.Fraction) for the GEMM, and numpy's
    fp64 matmul of dequantised operands;
  * brute force (sorting) for the token reorder, SciPy's expit for SiLU, and
    algebraic special cases (one expert, unit weight) for the combine.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden_e2m1():
    table = {}
    with open(os.path.join(GOLDEN, "e2m1_code_table.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            bits, val = line.split()
            table[int(bits, 2)] = float(val)
    assert len(table) == 16
    return table


def _golden_facts():
    facts = {}
    with open(os.path.join(GOLDEN, "format_facts.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                facts[k] = float(v)
    return facts


E2M1 = _golden_e2m1()
FACTS = _golden_facts()


def e4m3_value_ocp(b: int) -> float:
    """OCP FP8 E4M3FN: bias 7, subnormals, no inf, S.1111.111 = NaN."""
    s, e, m = (b >> 7) & 1, (b >> 3) & 15, b & 7
    if e == 15 and m == 7:
        return float("nan")
    v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
    return -v if s else v


def e2m1_by_boundaries(v: np.ndarray) -> np.ndarray:
    """Nearest-even E2M1 code as decision boundaries between neighbouring codes."""
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v.astype(np.float64))
    mags = [abs(E2M1[c]) for c in range(8)]
    code = np.zeros(v.shape, np.uint8)
    for c in range(1, 8):
        mid = (mags[c - 1] + mags[c]) / 2
        up = (a > mid) | ((a == mid) & (c % 2 == 0))
        code[up] = c
    return code | (np.signbit(v).astype(np.uint8) * 8)


def e4m3_by_frexp(t: np.ndarray) -> np.ndarray:
    """Nearest-even finite E4M3 byte of t >= 0 from its binary exponent."""
    t = np.asarray(t, dtype=np.float32).astype(np.float64)
    out = np.empty(t.shape, np.int64)
    sub = t < 2.0 ** -6
    out[sub] = np.rint(t[sub] * 512.0).astype(np.int64)  # grid 2^-9; 8 -> 0x08
    mant, ex = np.frexp(t[~sub])
    e = ex - 1
    f = np.rint((2 * mant - 1) * 8).astype(np.int64)
    carry = f == 8
    e = e + carry
    f = np.where(carry, 0, f)
    out[~sub] = np.minimum(((e + 7) << 3) | f, 0x7E)
    return out.astype(np.uint8)


def _rng(tag):
    return np.random.default_rng([20241202, tag])


# ---------------------------------------------------------------------------
# formats
# ---------------------------------------------------------------------------

def pin_e2m1_table(orc):
    for code, val in E2M1.items():
        got = orc.e2m1_value(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), (code, got, val)
        assert int(orc.e2m1_encode(np.float32(val))) == code, (code, val)
    assert max(abs(v) for v in E2M1.values()) == FACTS["e2m1_max"]


def pin_e2m1_ties(orc):
    # (value, code) worked by hand from the table and "ties to even, saturate".
    cases = [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
             (6.0, 7), (7.0, 7), (1e30, 7), (float("inf"), 7), (-0.1, 8), (-0.25, 8),
             (-0.26, 9), (0.2500001, 1), (2.9, 5), (-5.0001, 15), (-float("inf"), 15)]
    v = np.array([c[0] for c in cases], np.float32)
    got = orc.e2m1_encode(v)
    want = np.array([c[1] for c in cases], np.uint8)
    assert np.array_equal(got, want), list(zip(v, got, want))


def pin_e2m1_boundaries(orc):
    r = _rng(1)
    v = np.concatenate([
        (r.standard_normal(200000) * 3).astype(np.float32),
        (np.exp(r.uniform(-30, 10, 50000)) * r.choice([-1, 1], 50000)).astype(np.float32),
    ])
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(10))])
    v = np.concatenate([v, near, -near])
    assert np.array_equal(orc.e2m1_encode(v), e2m1_by_boundaries(v))


def pin_e4m3_roundtrip(orc):
    assert orc.e4m3_value(0x7E) == FACTS["e4m3_max"]
    assert math.isnan(orc.e4m3_value(0x7F)) and math.isnan(orc.e4m3_value(0xFF))
    for b in range(256):
        want = e4m3_value_ocp(b)
        got = orc.e4m3_value(b)
        if math.isnan(want):
            assert math.isnan(got), b
            continue
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (b, got, want)
        assert int(orc.e4m3_encode(np.float32(want))) == b, (b, want)
    assert FACTS["e2m1_max"] * FACTS["e4m3_max"] == FACTS["combined_range"]


def pin_e4m3_frexp(orc):
    r = _rng(2)
    t = np.exp(r.uniform(np.log(2.0 ** -12), np.log(2000.0), 300000)).astype(np.float32)
    vals = np.array([e4m3_value_ocp(b) for b in range(0x7F)], np.float64)
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)  # exact in FP32
    t = np.concatenate([t, mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
                        np.array([0, 448, 460, 464, 480, 1e20, 2.0 ** -10, 2.0 ** -11], np.float32)])
    assert np.array_equal(orc.e4m3_encode(t), e4m3_by_frexp(t))


def pin_e4m3_torch(orc):
    import torch
    r = _rng(3)
    t = np.exp(r.uniform(np.log(2.0 ** -12), np.log(448.0), 100000)).astype(np.float32)
    t = np.concatenate([t, np.array([0.0, 448.0, 2.0 ** -9, 2.0 ** -10], np.float32)])
    lib = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_encode(t), lib)


# ---------------------------------------------------------------------------
# block quantisation
# ---------------------------------------------------------------------------

def pin_block_worked(orc):
    # The table's 16 values, in code order; amax 6.  With g = 1, 2, 0.5 the
    # scale is g*6/6 = g (an E4M3 value), x*g/s = x, and the codes are 0..15.
    x = np.array([E2M1[c] for c in range(16)], np.float32)
    for g, sb_want in ((1.0, 0x38), (2.0, 0x40), (0.5, 0x30)):
        sb, codes = orc.quant_block16(x, g)
        assert sb == sb_want, (g, hex(sb))
        assert list(codes) == list(range(16)), (g, codes)
        q, sf = orc.quant_rows(x[None, :], np.array([g], np.float32))
        assert sf[0, 0] == sb_want
        assert list(q[0]) == [0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE], q
    # amax 7, g = 1: t = 7/6 -> nearest E4M3 is 1.125 (0x39); 7/1.125 saturates
    # to 6 (code 7); 0.25/1.125 = 0.22 -> 0; -1.125/1.125 = -1 -> code 10.
    x = np.zeros(16, np.float32)
    x[0], x[1], x[2] = 7.0, 0.25, -1.125
    sb, codes = orc.quant_block16(x, 1.0)
    assert sb == 0x39 and codes[0] == 7 and codes[1] == 0 and codes[2] == 10 and codes[3] == 0
    # an all-zero block: scale byte 0, every code 0
    sb, codes = orc.quant_block16(np.zeros(16, np.float32), 3.0)
    assert sb == 0 and not codes.any()


def pin_identity_2688(orc):
    # A tensor quantised with the global scale calibrated on its own amax
    # (scale = amax/2688, g = 1/scale): the block holding the amax element gets
    # scale 448 (0x7E) and that element gets the largest code, +-6.
    r = _rng(4)
    for trial in range(20):
        x = (r.standard_normal((8, 64)) * 10 ** r.uniform(-3, 3)).astype(np.float32)
        amax = np.float32(np.abs(x).max())
        scale = np.float32(amax / np.float32(FACTS["combined_range"]))
        g = np.float32(np.float32(1.0) / scale)
        q, sf = orc.quant_rows(x, np.full(8, g, np.float32))
        i, j = np.unravel_index(np.argmax(np.abs(x)), x.shape)
        assert sf[i, j // 16] == 0x7E, (trial, hex(sf[i, j // 16]))
        code = (q[i, j // 2] >> (4 * (j % 2))) & 15
        assert code == (15 if x[i, j] < 0 else 7), (trial, code)
        assert sf.max() <= 0x7E


def pin_block_invariances(orc):
    r = _rng(5)
    x = (r.standard_normal((64, 128)) * np.exp(r.uniform(-2, 2, (64, 1)))).astype(np.float32)
    g = np.exp(r.uniform(-3, 6, 64)).astype(np.float32)
    q, sf = orc.quant_rows(x, g)
    # sign symmetry: -x gives the same scales and codes with the sign bit set
    qn, sfn = orc.quant_rows(-x, g)
    assert np.array_equal(sf, sfn)
    assert np.array_equal(orc.unpack_codes(qn), orc.unpack_codes(q) ^ 8)
    # exact power-of-two rescaling of x against g changes nothing
    q2, sf2 = orc.quant_rows(x * np.float32(4.0), g / np.float32(4.0))
    assert np.array_equal(q, q2) and np.array_equal(sf, sf2)
    # each scale is the rounded g*amax/6, and each element is within half a
    # code step (at most 1, between 4 and 6) of x*g/s, or saturated at 6
    blocks = x.reshape(64, 8, 16)
    t = (np.abs(blocks).max(axis=2) * g[:, None]) / np.float32(6.0)
    assert np.array_equal(sf, e4m3_by_frexp(t.astype(np.float32)))
    s = np.array([e4m3_value_ocp(int(b)) for b in sf.ravel()]).reshape(sf.shape)
    vals = np.array([E2M1[c] for c in range(16)])[orc.unpack_codes(q)].reshape(64, 8, 16)
    target = blocks.astype(np.float64) * g[:, None, None] / s[:, :, None]
    err = np.abs(vals - np.clip(target, -6, 6))
    assert err.max() <= 1.0 + 1e-6


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------

def pin_route_bruteforce(orc):
    r = _rng(6)
    for T, k, E in ((1, 1, 1), (5, 2, 4), (37, 3, 9), (64, 8, 128)):
        ids = np.stack([r.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        offsets, perm = orc.route(ids, E)
        flat = ids.ravel()
        want = sorted(range(T * k), key=lambda f: (flat[f], f))
        assert list(perm) == want
        counts = np.bincount(flat, minlength=E)
        assert list(offsets) == [0] + list(np.cumsum(counts))


def pin_ue8m0(orc):
    """UE8M0 block scales.  Byte values against FP32 bit patterns (a float whose
    exponent field is b and mantissa 0 is 2^(b-127); 2^-127 is the subnormal
    0x00400000).  The encoding is the smallest power of two at or above t,
    checked with frexp on powers of two, their neighbours and log-uniform
    values.  Blocks: hand cases; against a numpy FP32 recomputation of
    x*g/s; no element saturates and the largest reaches at least 3; sign
    symmetry; the zero block."""
    for b in range(1, 255):
        assert orc.ue8m0_value(b) == float(np.uint32(b << 23).view(np.float32)), b
    assert orc.ue8m0_value(0) == float(np.uint32(0x00400000).view(np.float32))
    assert math.isnan(orc.ue8m0_value(255))

    def by_frexp(t):
        if not t > 2.0 ** -127:
            return 0
        if math.isinf(t):
            return 254
        m, e = math.frexp(t)  # t = m * 2^e, 0.5 <= m < 1
        return min((e - 1 if m == 0.5 else e) + 127, 254)

    r = _rng(31)
    ts = [0.0, float(np.finfo(np.float32).max), float("inf"), 2.0 ** -149, 2.0 ** -127, 2.0 ** 127]
    for k in range(-149, 128):
        p2 = np.float32(2.0) ** np.float32(k) if k > -127 else np.float32(2.0 ** k)
        ts += [float(p2), float(np.nextafter(p2, np.float32(np.inf))), float(np.nextafter(p2, np.float32(0)))]
    with np.errstate(over="ignore"):  # values beyond FP32 become inf, which is a case too
        ts += list(np.exp(r.uniform(-100, 100, 4000)).astype(np.float32).astype(float))
    for t in ts:
        assert orc.ue8m0_encode(t) == by_frexp(float(np.float32(t))), t

    table = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, 0, -0.5, -1, -1.5, -2, -3, -4, -6], np.float32)
    sb, codes = orc.quant_block16(table, 1.0, ue8m0=True)
    assert sb == 127 and codes.tolist() == [0, 1, 2, 3, 4, 5, 6, 7, 0, 9, 10, 11, 12, 13, 14, 15]
    sb, codes = orc.quant_block16(table * 2, 1.0, ue8m0=True)
    assert sb == 128 and codes.tolist() == [0, 1, 2, 3, 4, 5, 6, 7, 0, 9, 10, 11, 12, 13, 14, 15]
    sb, codes = orc.quant_block16(np.full(16, 7.0, np.float32), 1.0, ue8m0=True)
    assert sb == 128 and np.all(codes == 6)  # t = 7/6 -> s = 2; 3.5 ties to the even code, 4.0
    sb, codes = orc.quant_block16(np.zeros(16, np.float32), 3.0, ue8m0=True)
    assert sb == 0 and np.all(codes == 0)
    for _ in range(3000):
        x = (r.standard_normal(16) * np.exp(r.uniform(-20, 20))).astype(np.float32)
        g = np.float32(np.exp(r.uniform(-10, 10)))
        sb, codes = orc.quant_block16(x, g, ue8m0=True)
        amax = np.float32(np.abs(x).max())
        t = np.float32(np.float32(g * amax) / np.float32(6.0))
        s = orc.ue8m0_value(sb)
        assert s >= t and (sb == 0 or s / 2 < t)
        y = (x * g).astype(np.float32)
        q = (y.astype(np.float64) / s).astype(np.float32)
        assert np.array_equal(codes, orc.e2m1_encode(q))
        vals = orc.e2m1_values(codes)
        assert np.all(np.abs(vals) <= 6)
        if sb > 0:
            assert np.abs(vals).max() >= 3
        sb2, codes2 = orc.quant_block16(-x, g, ue8m0=True)
        assert sb2 == sb and np.array_equal(codes2, codes ^ 8)


def _bf16_round_fraction(v: Fraction) -> Fraction:
    """Nearest BF16 value (8 significant bits, ties to even), by exact
    rational arithmetic."""
    if v == 0:
        return Fraction(0)
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    step = Fraction(2) ** (e - 7)          # spacing of 8-bit significands at this binade
    q, rem = divmod(a, step)
    if rem * 2 > step or (rem * 2 == step and q % 2 == 1):
        q += 1
    return (q * step) if v > 0 else -(q * step)


def pin_w4a16(orc):
    """The W4A16 layer on a tiny case against exact rational arithmetic: the
    weights decoded from the page's E2M1 table (golden file) and an E4M3
    formula written here, times weight_scale_2; both GEMMs and the combine as
    exact sums; h = SiLU(gate) * up in double, rounded to BF16 by a rational
    round-to-nearest-even.  Catches a dropped scale, swapped gate/up,
    transposed operands, an h that skips its BF16 rounding and wrong weights
    in the combine."""
    r = _rng(41)
    E, H, I, T, k = 2, 32, 32, 3, 2

    class W:
        pass

    W.E, W.H, W.I = E, H, I
    W.w13_q = r.integers(0, 256, (E, 2 * I, H // 2)).astype(np.uint8)
    W.w13_sf = r.integers(0x28, 0x48, (E, 2 * I, H // 16)).astype(np.uint8)
    W.w13_scale2 = np.array([0.75, 1.0 / 3.0], np.float32)
    W.w2_q = r.integers(0, 256, (E, H, I // 2)).astype(np.uint8)
    W.w2_sf = r.integers(0x28, 0x48, (E, H, I // 16)).astype(np.uint8)
    W.w2_scale2 = np.array([0.5, 1.25], np.float32)
    x = (r.standard_normal((T, H)) * 0.25).astype(np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncated to BF16 bits: any BF16 input will do
    ids = np.array([[0, 1], [1, 0], [0, 1]], np.int32)
    tw = np.array([[0.75, 0.25], [0.5, 0.5], [1.0, 0.0]], np.float32)
    got = orc.moe_forward_w4a16(xb, ids, tw, W)

    def e4m3(b):
        ex, m = (b >> 3) & 15, b & 7
        return Fraction(m, 512) if ex == 0 else Fraction(8 + m, 8) * Fraction(2) ** (ex - 7)

    def weights(q, sf, s2):
        N, K = q.shape[0], q.shape[1] * 2
        out = [[Fraction(0)] * K for _ in range(N)]
        for n in range(N):
            for kk in range(K):
                byte = int(q[n, kk // 2])
                code = byte & 15 if kk % 2 == 0 else byte >> 4
                out[n][kk] = Fraction(E2M1[code]) * e4m3(int(sf[n, kk // 16])) * Fraction(float(s2))
        return out

    w13 = [weights(W.w13_q[e], W.w13_sf[e], W.w13_scale2[e]) for e in range(E)]
    w2 = [weights(W.w2_q[e], W.w2_sf[e], W.w2_scale2[e]) for e in range(E)]
    xf = [[Fraction(float(np.uint32(int(b) << 16).view(np.float32))) for b in row] for row in xb]
    for t in range(T):
        acc = [Fraction(0)] * H
        for j in range(k):
            e, wt = int(ids[t, j]), Fraction(float(tw[t, j]))
            y1 = [sum(xf[t][kk] * w13[e][n][kk] for kk in range(H)) for n in range(2 * I)]
            h = []
            for i in range(I):
                g, u = float(y1[i]), float(y1[I + i])
                h.append(_bf16_round_fraction(Fraction(g / (1.0 + math.exp(-g)) * u)))
            for n in range(H):
                acc[n] += wt * sum(h[i] * w2[e][n][i] for i in range(I))
        want = np.array([float(a) for a in acc])
        assert np.allclose(got["out"][t], want, rtol=1e-12, atol=1e-300), (t, np.abs(got["out"][t] - want).max())


def pin_router(orc):
    """Router pins: k = E is SciPy's softmax in the stable descending order of the
    logits; for k < E the renormalised weights are the softmax of the selected
    logits (an identity of renormalisation, checked with SciPy); hand cases for
    ties, equal logits and a dominant logit; brute-force selection on tiny
    inputs; shift invariance."""
    from scipy.special import softmax
    r = _rng(21)
    lg = r.standard_normal((16, 9)).astype(np.float32)
    ids, w = orc.router(lg, 9)
    assert np.array_equal(ids, np.argsort(-lg, axis=1, kind="stable"))
    ref = softmax(lg.astype(np.float64), axis=1)
    assert np.allclose(w, np.take_along_axis(ref, ids, axis=1), rtol=2e-7, atol=0)
    for k in (1, 3, 5):
        ids, w = orc.router(lg, k)
        sub = softmax(np.take_along_axis(lg, ids, axis=1).astype(np.float64), axis=1)
        assert np.allclose(w, sub, rtol=2e-7, atol=0)
        assert np.all(np.diff(w, axis=1) <= 0)
    # ties go to the lower index; equal logits share the weight exactly
    ids, w = orc.router(np.array([[0.0, 5.0, 5.0, 1.0]], np.float32), 2)
    assert ids.tolist() == [[1, 2]] and w.tolist() == [[0.5, 0.5]]
    ids, w = orc.router(np.zeros((3, 8), np.float32), 4)
    assert ids.tolist() == [[0, 1, 2, 3]] * 3 and np.all(w == 0.25)
    # a dominant logit takes all the weight
    big = r.standard_normal((1, 32)).astype(np.float32)
    big[0, 17] = 60.0
    ids, w = orc.router(big, 1)
    assert ids.tolist() == [[17]] and w.tolist() == [[1.0]]
    # logits whose fp64 probabilities tie are ordered by the logits themselves
    ids, _ = orc.router(np.array([[0.0, 1e-30, 0.0, 2e-30]], np.float32), 2)
    assert ids.tolist() == [[3, 1]]
    # brute-force selection on tiny inputs with many duplicate values
    for _ in range(50):
        E = int(r.integers(1, 7))
        k = int(r.integers(1, E + 1))
        row = r.integers(-2, 3, E).astype(np.float32)
        ids, _ = orc.router(row[None, :], k)
        assert ids[0].tolist() == sorted(range(E), key=lambda e: (-row[e], e))[:k]
    # shifting every logit changes nothing but rounding
    ids0, w0 = orc.router(lg, 4)
    ids1, w1 = orc.router(lg + np.float32(2.0), 4)
    assert np.array_equal(ids0, ids1) and np.allclose(w0, w1, rtol=1e-6, atol=0)


# ---------------------------------------------------------------------------
# GEMM, activation, combine
# ---------------------------------------------------------------------------

def _gemm_fraction(aq, asf, ga, wq, wsf, gw):
    def row_values(q, sf):
        vals = []
        for i in range(len(q) * 2):
            code = (int(q[i // 2]) >> (4 * (i % 2))) & 15
            vals.append(Fraction(E2M1[code]) * Fraction(e4m3_value_ocp(int(sf[i // 16]))))
        return vals
    A = [row_values(aq[m], asf[m]) for m in range(aq.shape[0])]
    W = [row_values(wq[n], wsf[n]) for n in range(wq.shape[0])]
    y = np.empty((len(A), len(W)))
    for m, a in enumerate(A):
        for n, w in enumerate(W):
            y[m, n] = float(sum(p * q for p, q in zip(a, w)) / (Fraction(float(ga[m])) * Fraction(float(gw))))
    return y


def _tiny_operands(r, M, N, K):
    x = r.standard_normal((M, K)).astype(np.float32)
    w = (r.standard_normal((N, K)) * 0.02).astype(np.float32)
    ga = np.exp(r.uniform(-1, 6, M)).astype(np.float32)
    gw = np.float32(np.exp(r.uniform(3, 9)))
    aq, asf = orc_quant(x, ga)
    wq, wsf = orc_quant(w, np.full(N, gw, np.float32))
    return aq, asf, ga, wq, wsf, gw


_ORC = None


def orc_quant(x, g):
    return _ORC.quant_rows(x, g)


def pin_gemm_fraction(orc):
    global _ORC
    _ORC = orc
    r = _rng(7)
    aq, asf, ga, wq, wsf, gw = _tiny_operands(r, 3, 5, 48)
    y = orc.gemm(aq, asf, ga, wq, wsf, gw)
    want = _gemm_fraction(aq, asf, ga, wq, wsf, gw)
    assert np.allclose(y, want, rtol=1e-15, atol=0), (y, want)


def pin_gemm_fp64(orc):
    global _ORC
    _ORC = orc
    r = _rng(8)
    aq, asf, ga, wq, wsf, gw = _tiny_operands(r, 17, 40, 256)

    def deq(q, sf, g):
        codes = np.empty((q.shape[0], q.shape[1] * 2), np.int64)
        codes[:, 0::2], codes[:, 1::2] = q & 15, q >> 4
        v = np.array([E2M1[c] for c in range(16)])[codes]
        s = np.array([e4m3_value_ocp(b) for b in range(256)])[sf.astype(np.int64)]
        return v * np.repeat(s, 16, axis=1) / np.asarray(g, np.float64).reshape(-1, 1)

    want = deq(aq, asf, ga) @ deq(wq, wsf, np.full(wq.shape[0], gw)).T
    y = orc.gemm(aq, asf, ga, wq, wsf, gw)
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def _ue8m0_fraction(b: int) -> Fraction:
    # UE8M0 byte b encodes 2^(b - 127) (255 is NaN and never produced)
    return Fraction(2) ** (int(b) - 127)


def pin_gemm_ue8m0_fraction(orc):
    """The UE8M0 GEMM against exact rational arithmetic, with global scales
    spread over 2^-60 .. 2^60 so that the block scale bytes lie far from the
    bias and a wrong bias, a dropped scale or a swapped nibble shows."""
    r = _rng(21)
    M, N, K = 3, 4, 48
    x = r.standard_normal((M, K)).astype(np.float32)
    w = (r.standard_normal((N, K)) * 0.02).astype(np.float32)
    ga = np.exp2(r.uniform(-60, 60, M)).astype(np.float32)
    gw = np.float32(np.exp2(r.uniform(-40, 40)))
    aq, asf = orc.quant_rows(x, ga, ue8m0=True)
    wq, wsf = orc.quant_rows(w, np.full(N, gw, np.float32), ue8m0=True)
    assert asf.min() < 100 or asf.max() > 150  # far from the bias
    y = orc.gemm_ue8m0(aq, asf, ga, wq, wsf, gw)

    def row_values(q, sf):
        return [Fraction(E2M1[(int(q[i // 2]) >> (4 * (i % 2))) & 15]) * _ue8m0_fraction(sf[i // 16])
                for i in range(len(q) * 2)]

    for m in range(M):
        a = row_values(aq[m], asf[m])
        for n in range(N):
            b = row_values(wq[n], wsf[n])
            want = sum(p * q for p, q in zip(a, b)) / (Fraction(float(ga[m])) * Fraction(float(gw)))
            assert abs(y[m, n] - float(want)) <= 1e-15 * abs(float(want)) + 1e-300, (m, n, y[m, n], float(want))


def pin_gemm_ue8m0_matches_e4m3(orc):
    """On block scales that are powers of two inside E4M3's range (2^-9 ..
    2^8), the same operands written with E4M3 and with UE8M0 scale bytes give
    the same GEMM: the UE8M0 GEMM against the rationally pinned E4M3 one.
    The bytes come from test-side encoders of 2^k."""
    r = _rng(22)
    M, N, K = 9, 7, 96

    def e4m3_pow2(k):
        return ((k + 7) << 3) if k >= -6 else (1 << (k + 9))

    ka = r.integers(-9, 9, (M, K // 16))
    kw = r.integers(-9, 9, (N, K // 16))
    aq = r.integers(0, 256, (M, K // 2)).astype(np.uint8)
    wq = r.integers(0, 256, (N, K // 2)).astype(np.uint8)
    ga = np.exp(r.uniform(-2, 2, M)).astype(np.float32)
    gw = np.float32(3.0)
    enc = np.vectorize(e4m3_pow2)
    assert all(e4m3_value_ocp(e4m3_pow2(k)) == 2.0 ** k for k in range(-9, 9))
    y_e4 = orc.gemm(aq, enc(ka).astype(np.uint8), ga, wq, enc(kw).astype(np.uint8), gw)
    y_ue = orc.gemm_ue8m0(aq, (ka + 127).astype(np.uint8), ga, wq, (kw + 127).astype(np.uint8), gw)
    assert np.allclose(y_ue, y_e4, rtol=1e-15, atol=1e-15 * np.abs(y_e4).max())


def pin_silu_mul(orc):
    from scipy.special import expit
    r = _rng(9)
    I = 24
    y1 = r.standard_normal((7, 2 * I)) * 6
    y1[0, :I] = 0.0
    y1[1, :I] = 800.0
    y1[2, :I] = -800.0
    h = orc.silu_mul(y1)
    gate, up = y1[:, :I], y1[:, I:]
    want = (gate * expit(gate) * up).astype(np.float32)
    assert np.allclose(h, want, rtol=2e-7, atol=1e-30)
    assert not h[0].any() and np.array_equal(h[1], (800.0 * up[1]).astype(np.float32))
    assert np.all(np.abs(h[2]) == 0)


def _small_weights(orc, r, E, H, I):
    W = orc.Weights(E, H, I)
    for e in range(E):
        w13 = (r.standard_normal((2 * I, H)) * 0.02).astype(np.float32)
        w2 = (r.standard_normal((H, I)) * 0.02).astype(np.float32)
        for name, w in (("w13", w13), ("w2", w2)):
            bits = (w.view(np.uint32) >> 16).astype(np.uint16)  # truncation: any BF16 input will do
            q, sf, s2 = orc.quantize_weight(bits)
            getattr(W, name + "_q")[e], getattr(W, name + "_sf")[e] = q, sf
            getattr(W, name + "_scale2")[e] = s2
    W.w13_input_scale = np.exp(r.uniform(-9, -6, E)).astype(np.float32)
    W.w2_input_scale = np.exp(r.uniform(-9, -6, E)).astype(np.float32)
    return W


def pin_combine_special(orc):
    r = _rng(10)
    E, H, I, T = 3, 32, 16, 6
    W = _small_weights(orc, r, E, H, I)
    x = (r.standard_normal((T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    # one expert per token with weight 1: out is that row's w2 output
    ids = r.integers(0, E, (T, 1)).astype(np.int32)
    res = orc.moe_forward(x, ids, np.ones((T, 1), np.float32), W)
    t_of = res["perm"][res["rows"]]
    assert np.array_equal(res["out"][t_of], res["y2"])
    # two experts: out = w0*y(t,0) + w1*y(t,1), and out is linear in the weights
    ids2 = np.stack([r.choice(E, 2, replace=False) for _ in range(T)]).astype(np.int32)
    w = r.uniform(0, 1, (T, 2)).astype(np.float32)
    a = orc.moe_forward(x, ids2, w, W)
    b = orc.moe_forward(x, ids2, (w * np.float32(2.0)).astype(np.float32), W)
    assert np.allclose(b["out"], 2 * a["out"], rtol=1e-15, atol=0)
    f = a["perm"][a["rows"]]
    want = np.zeros((T, H))
    for row, ff in enumerate(f):
        want[ff // 2] += float(w.ravel()[ff]) * a["y2"][row]
    assert np.allclose(a["out"], want, rtol=1e-14, atol=0)


def pin_forward_stepwise(orc):
    """Each GEMM stage of the oracle's forward against an fp64 numpy matmul of
    the dequantised operands (test-side decoders), and gate/up order against
    SciPy's expit."""
    from scipy.special import expit
    r = _rng(11)
    E, H, I, T, k = 2, 64, 32, 8, 2
    W = _small_weights(orc, r, E, H, I)
    x = (r.standard_normal((T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    ids = np.stack([r.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = r.uniform(0, 1, (T, k)).astype(np.float32)
    res = orc.moe_forward(x, ids, w, W)
    tab = np.array([E2M1[c] for c in range(16)])
    stab = np.array([e4m3_value_ocp(b) if b != 0x7F and b != 0xFF else 0 for b in range(256)])

    def deq(q, sf, g):
        codes = np.empty((q.shape[0], q.shape[1] * 2), np.int64)
        codes[:, 0::2], codes[:, 1::2] = q & 15, q >> 4
        return tab[codes] * np.repeat(stab[sf.astype(np.int64)], 16, axis=1) / np.float64(g)

    g1 = np.float32(1) / W.w13_input_scale
    g2 = np.float32(1) / W.w2_input_scale
    for e in range(E):
        sel = res["row_expert"][res["rows"]] == e
        a1 = deq(res["a1q"][sel], res["sf1"][sel], g1[e])
        w13 = deq(W.w13_q[e], W.w13_sf[e], np.float32(1) / W.w13_scale2[e])
        y1 = a1 @ w13.T
        gate, up = y1[:, :I], y1[:, I:]
        assert np.allclose(res["h"][sel], (gate * expit(gate) * up).astype(np.float32), rtol=1e-6,
                           atol=1e-6 * np.abs(res["h"][sel]).max())
        a2 = deq(res["a2q"][sel], res["sf2"][sel], g2[e])
        w2 = deq(W.w2_q[e], W.w2_sf[e], np.float32(1) / W.w2_scale2[e])
        assert np.allclose(res["y2"][sel], a2 @ w2.T, rtol=1e-12, atol=1e-12 * np.abs(res["y2"]).max())


def pin_forward_stepwise_ue8m0(orc):
    """The forward with UE8M0 block scales throughout: every scale byte of a1
    and a2 is the smallest power of two at or above fl(fl(g*amax)/6), and each
    GEMM stage matches an fp64 numpy matmul of operands decoded on the test
    side (2^(b - 127) scales)."""
    from scipy.special import expit
    r = _rng(23)
    E, H, I, T, k = 2, 64, 32, 8, 2
    W = orc.Weights(E, H, I)
    W.ue8m0 = True
    for e in range(E):
        for name, shape in (("w13", (2 * I, H)), ("w2", (H, I))):
            wv = (r.standard_normal(shape) * 0.02).astype(np.float32)
            q, sf, s2 = orc.quantize_weight((wv.view(np.uint32) >> 16).astype(np.uint16), ue8m0=True)
            getattr(W, name + "_q")[e], getattr(W, name + "_sf")[e] = q, sf
            getattr(W, name + "_scale2")[e] = s2
    W.w13_input_scale = np.exp(r.uniform(-9, -6, E)).astype(np.float32)
    W.w2_input_scale = np.exp(r.uniform(-9, -6, E)).astype(np.float32)
    x = (r.standard_normal((T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    ids = np.stack([r.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = r.uniform(0, 1, (T, k)).astype(np.float32)
    res = orc.moe_forward(x, ids, w, W)
    tab = np.array([E2M1[c] for c in range(16)])

    def deq(q, sf, g):
        codes = np.empty((q.shape[0], q.shape[1] * 2), np.int64)
        codes[:, 0::2], codes[:, 1::2] = q & 15, q >> 4
        return tab[codes] * np.repeat(np.exp2(sf.astype(np.float64) - 127), 16, axis=1) / np.float64(g)

    def check_scales(vals, sf, g):
        # vals [rows, K] FP32 values that were quantised with global scale g per row
        for i in range(vals.shape[0]):
            for b in range(sf.shape[1]):
                amax = np.float32(np.abs(vals[i, 16 * b:16 * b + 16]).max())
                t = np.float32(np.float32(np.float32(g[i]) * amax) / np.float32(6))
                if t == 0:
                    continue
                s = 2.0 ** (int(sf[i, b]) - 127)
                assert s >= t and s / 2 < t, (i, b, s, t)

    xf = (x.astype(np.uint32) << 16).view(np.float32)
    g1 = np.float32(1) / W.w13_input_scale
    g2 = np.float32(1) / W.w2_input_scale
    rows = res["rows"]
    re = res["row_expert"][rows]
    check_scales(xf[res["perm"][rows] // k], res["sf1"], g1[re])
    check_scales(res["h"], res["sf2"], g2[re])
    for e in range(E):
        sel = re == e
        a1 = deq(res["a1q"][sel], res["sf1"][sel], g1[e])
        w13 = deq(W.w13_q[e], W.w13_sf[e], np.float32(1) / W.w13_scale2[e])
        y1 = a1 @ w13.T
        gate, up = y1[:, :I], y1[:, I:]
        assert np.allclose(res["h"][sel], (gate * expit(gate) * up).astype(np.float32), rtol=1e-6,
                           atol=1e-6 * np.abs(res["h"][sel]).max())
        a2 = deq(res["a2q"][sel], res["sf2"][sel], g2[e])
        w2 = deq(W.w2_q[e], W.w2_sf[e], np.float32(1) / W.w2_scale2[e])
        assert np.allclose(res["y2"][sel], a2 @ w2.T, rtol=1e-12, atol=1e-12 * np.abs(res["y2"]).max())


# ---------------------------------------------------------------------------
# composition: routed rows in permuted order, token subsets
# ---------------------------------------------------------------------------

def _order_by_sort(ids):
    """The permuted order by brute force: flat routed rows f = t*k + j sorted
    by (expert, f) (the page's reorder by expert; stable within an expert)."""
    flat = np.asarray(ids).ravel()
    return sorted(range(flat.size), key=lambda f: (int(flat[f]), f))


def _row_by_blocks(orc, xrow, g, ue8m0=False):
    """One row quantised block by block with the pinned single-block routine,
    codes packed two per byte, element 2i in the low nibble."""
    H = xrow.size
    q = np.zeros(H // 2, np.uint8)
    sf = np.zeros(H // 16, np.uint8)
    for b in range(H // 16):
        sb, codes = orc.quant_block16(xrow[16 * b:16 * b + 16], g, ue8m0=ue8m0)
        sf[b] = sb
        c = np.asarray(codes, np.uint8)
        q[8 * b:8 * b + 8] = c[0::2] | (c[1::2] << 4)
    return q, sf


def _ragged_routing(r, T, k, E, skip=()):
    """Distinct experts per token, some experts left empty (ragged groups)."""
    allowed = np.array([e for e in range(E) if e not in skip])
    return np.stack([r.choice(allowed, k, replace=False) for _ in range(T)]).astype(np.int32)


def pin_quantize_experts_rows(orc):
    """Routed-row quantisation: permuted row p is token perm[p] // k
    quantised with the global scale fl(1/input_scale[e]) of the expert e that
    row belongs to (page "Gemma 4 NVFP4 MoE 空输出", MoE section: the expert
    index selects SFScale; §矩阵融合 "MoE FFN": rows reordered by expert).
    The permutation, each row's token and each row's scale are recomputed
    here from the routing alone; T, k are chosen so that f % k and f // k
    differ for most rows."""
    r = _rng(31)
    for ue in (False, True):
        for T, k, E, skip in ((7, 3, 5, (2,)), (11, 2, 6, (0, 4)), (3, 1, 2, ())):
            H = 48
            x = (r.standard_normal((T, H)).astype(np.float32) * np.float32(3)).view(np.uint32)
            x = (x >> 16).astype(np.uint16)
            # one token made large so a wrong token shows in every scale byte
            x[T // 2] = ((x[T // 2].astype(np.uint32) << 16).view(np.float32) * np.float32(64)).view(np.uint32) >> 16
            ids = _ragged_routing(r, T, k, E, skip)
            scales = np.exp(r.uniform(-4, 2, E)).astype(np.float32)
            q, sf, offsets, perm = orc.quantize_experts(x, ids, scales, E, ue8m0=ue)
            order = _order_by_sort(ids)
            assert list(perm) == order
            flat = ids.ravel()
            assert list(offsets) == [0] + list(np.cumsum(np.bincount(flat, minlength=E)))
            xf = (x.astype(np.uint32) << 16).view(np.float32)
            for p, f in enumerate(order):
                e = int(flat[f])
                g = np.float32(np.float32(1.0) / scales[e])
                wq, wsf = _row_by_blocks(orc, xf[f // k], g, ue8m0=ue)
                assert np.array_equal(q[p], wq), (ue, T, k, p)
                assert np.array_equal(sf[p], wsf), (ue, T, k, p)


def pin_forward_token_subset(orc):
    """The forward restricted to a token subset S (a test-size device of the
    oracle: the full-size checks compute sampled tokens only).  Restoring the
    token order and summing with the routing weights (page "Gemma 4 NVFP4 MoE
    空输出", §矩阵融合 pipeline figure) is per token, so out on S must equal
    the full run's out on S exactly and be 0 elsewhere; the computed rows must
    be exactly the permuted rows whose token is in S, each intermediate row
    equal to the full run's row; and the a1 codes of every row must be its
    token's row quantised with its expert's scale."""
    r = _rng(32)
    E, H, I, T, k = 4, 32, 16, 9, 3
    W = _small_weights(orc, r, E, H, I)
    x = (r.standard_normal((T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    ids = _ragged_routing(r, T, k, E)
    w = r.uniform(0.1, 1, (T, k)).astype(np.float32)
    full = orc.moe_forward(x, ids, w, W)
    order = _order_by_sort(ids)
    assert list(full["perm"]) == order
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    g1 = (np.float32(1) / W.w13_input_scale).astype(np.float32)
    flat = ids.ravel()
    for p, f in enumerate(order):
        wq, wsf = _row_by_blocks(orc, xf[f // k], g1[flat[f]])
        assert np.array_equal(full["a1q"][p], wq) and np.array_equal(full["sf1"][p], wsf), p
    for S in ([0], [T - 1, 2], [1, 4, 5, 8], list(range(T))):
        sub = orc.moe_forward(x, ids, w, W, tokens=S)
        want_rows = [p for p, f in enumerate(order) if f // k in S]
        assert list(sub["rows"]) == want_rows, S
        keep = np.zeros(T, bool)
        keep[S] = True
        assert np.array_equal(sub["out"][keep], full["out"][keep]), S
        assert not sub["out"][~keep].any(), S
        for name in ("a1q", "sf1", "h", "a2q", "sf2", "y2"):
            assert np.array_equal(sub[name], full[name][want_rows]), (S, name)
    # the W4A16 forward's subset path, likewise
    full16 = orc.moe_forward_w4a16(x, ids, w, W)
    for S in ([3], [0, 7, 8]):
        sub = orc.moe_forward_w4a16(x, ids, w, W, tokens=S)
        want_rows = [p for p, f in enumerate(order) if f // k in S]
        assert list(sub["rows"]) == want_rows, S
        keep = np.zeros(T, bool)
        keep[S] = True
        assert np.array_equal(sub["out"][keep], full16["out"][keep]) and not sub["out"][~keep].any(), S
        assert np.array_equal(sub["h"], full16["h"][want_rows]), S


# ---------------------------------------------------------------------------
# validation, residual + RMSNorm
# ---------------------------------------------------------------------------

def pin_validate(orc):
    good = [1e-3, 0.5, 1.0, 2.0 ** 100, 2.0 ** -120]
    bad = [0.0, -1.0, float("nan"), float("inf"), -float("inf"), 1e-40, 2.0 ** 127]
    for v in good:
        assert orc.validate_scales(np.array([v], np.float32)) == (0, -1), v
    for v in bad:
        assert orc.validate_scales(np.array([v], np.float32)) == (1, 0), v
    s = np.ones(10, np.float32)
    s[[3, 7]] = np.nan
    assert orc.validate_scales(s) == (2, 3)
    written = np.ones(10, np.uint8)
    written[5] = 0
    assert orc.validate_scales(np.ones(10, np.float32), written) == (1, 5)
    sent = np.ones(4, np.float32)
    sent.view(np.uint32)[2] = 0x7FC00000
    assert orc.validate_scales(sent) == (1, 2)


def pin_rmsnorm(orc):
    r = _rng(12)
    T, H = 5, 96
    x = (r.standard_normal((T, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    out = r.standard_normal((T, H)).astype(np.float32)
    # last row: tiny residual (mean square ~ eps), so eps visibly matters
    x[-1] = 0
    out[-1] = (out[-1] * np.float32(1e-3)).astype(np.float32)
    xn = orc.residual_rmsnorm(x, out, 1e-6)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    res = xf + out.astype(np.float64)
    want = res / np.sqrt((res ** 2).mean(axis=1, keepdims=True) + 1e-6)
    got = (xn.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # nearest BF16: within half a BF16 step (2^-8 relative) of the exact value
    ulp = 2.0 ** (np.floor(np.log2(np.abs(want))) - 7)
    assert np.all(np.abs(got - want) <= ulp / 2 * (1 + 1e-12))
    one = orc.residual_rmsnorm(np.zeros((1, 4), np.uint16), np.full((1, 4), 3.0, np.float32), 0.0)
    assert np.all(one == 0x3F80)  # 3 / sqrt(9) = 1.0


ALL_PINS = [
    pin_e2m1_table, pin_e2m1_ties, pin_e2m1_boundaries, pin_e4m3_roundtrip, pin_e4m3_frexp,
    pin_e4m3_torch, pin_block_worked, pin_identity_2688, pin_block_invariances,
    pin_route_bruteforce, pin_gemm_fraction, pin_gemm_fp64, pin_silu_mul, pin_combine_special,
    pin_forward_stepwise, pin_validate, pin_rmsnorm, pin_router, pin_ue8m0, pin_w4a16,
    pin_gemm_ue8m0_fraction, pin_gemm_ue8m0_matches_e4m3, pin_forward_stepwise_ue8m0,
    pin_quantize_experts_rows, pin_forward_token_subset,
]
