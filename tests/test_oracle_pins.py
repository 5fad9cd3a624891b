"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test names the fact it checks.  None of them re-types an oracle formula
and compares it with itself: they use values printed on the pages, closed
forms, library routines on special cases, brute force and invariants.
"""

import math
import os

import numpy as np
import pytest

from mixed_precision_bit_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F16MAX = 65504.0


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16(x):
    return synth.from_bits(synth.to_bits(np.asarray(x, np.float32), synth.BF16), synth.BF16)


# ----------------------------------------------------------------- effective bits
def test_avg_bits_table(orc):
    """VeloxQuant-MLX docs, "Tuning avg_bits" table and "Effective bit-width"."""
    rows = [l.split() for l in open(os.path.join(GOLDEN, "avg_bits_table.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 4
    for hf, hi, lo, bits, comp in rows:
        got = orc.avg_bits(float(hf), int(hi), int(lo))
        assert got == pytest.approx(float(bits), abs=1e-12)
        assert round(16.0 / got, 1) == pytest.approx(float(comp))
    assert orc.avg_bits(0.25, 4, 2) == 2.5 and 16 / 2.5 == 6.4


def test_page_bytes_and_real_bits(orc):
    """Fixed-size page blob: 3072 + 9*n_hi bytes; 3360/3216/3072 at n_hi=32/16/0,
    i.e. 3.28/3.14/3.0 bits per K+V element with fp16 metadata."""
    assert orc.page_bytes(32) == 3360 and orc.page_bytes(16) == 3216 and orc.page_bytes(0) == 3072
    for n in range(0, 129, 16):
        assert orc.page_bytes(n) == 3072 + 9 * n
        assert orc.page_bytes(n) % 16 == 0
    for bad in (-16, 8, 144, 130):
        assert orc.page_bytes(bad) == -1
    per_elem = {n: orc.page_bytes(n) * 8 / (2 * 32 * 128) for n in (32, 16, 0)}
    assert round(per_elem[32], 2) == 3.28 and round(per_elem[16], 2) == 3.14
    assert per_elem[0] == 3.0


# ----------------------------------------------------------------- number formats
def test_f16_rounding_matches_numpy(orc):
    """fp32 -> fp16 round-to-nearest-even, subnormals and overflow, against numpy."""
    r = _rng(1)
    vals = np.concatenate([
        r.standard_normal(4000).astype(np.float32) * np.float32(10.0) ** r.integers(-9, 6, 4000),
        np.array([0.0, -0.0, 65504, 65519.9, 65520, 65536, 6.1035156e-05, 5.96e-08, 2.98e-08,
                  2.9802322e-08, 1e-30, -1e-30, np.inf, -np.inf, 1.00048828125, 1.000732421875],
                 np.float32)])
    for x in vals:
        with np.errstate(over="ignore"):
            want = int(np.float32(x).astype(np.float16).view(np.uint16))
        assert orc.f32_to_f16_bits(float(x)) == want, x
    for h in range(0, 1 << 16, 7):
        f = np.uint16(h).view(np.float16)
        if np.isnan(f):
            continue
        assert orc.f16_bits_to_f32(h) == np.float32(f)


# ----------------------------------------------------------------- statistics
def test_tree_sum_order(orc):
    """Tree order, hand-derived: x0 = 2^24, x1 = x17 = 1.  Tree pairs x1 with x17
    first, so the total is 2^24 + 2; a left-to-right sum gives 2^24."""
    x = np.zeros(32, np.float32)
    x[0], x[1], x[17] = 2.0 ** 24, 1.0, 1.0
    assert float(orc.tree_sum(x)) == 2.0 ** 24 + 2
    seq = np.float32(0)
    for v in x:
        seq = np.float32(seq + v)
    assert float(seq) == 2.0 ** 24
    ints = _rng(2).integers(-1000, 1000, 32).astype(np.float32)
    assert float(orc.tree_sum(ints)) == float(ints.sum(dtype=np.float64))


def test_variance_vs_two_pass(orc):
    """sum/sumsq variance estimate against an fp64 two-pass variance."""
    r = _rng(3)
    for _ in range(200):
        x = _bf16(r.standard_normal(32) * math.exp(r.standard_normal()) + r.standard_normal())
        s = orc.tree_sum(x)
        sq = orc.tree_sum((x * x).astype(np.float32))
        v = float(orc.variance(s, sq, 32.0))
        ref = float(np.var(x.astype(np.float64)))
        assert abs(v - ref) <= 1e-5 * float(np.mean(x.astype(np.float64) ** 2)) + 1e-30
    c = np.full(32, 0.375, np.float32)
    assert float(orc.variance(orc.tree_sum(c), orc.tree_sum(c * c), 32.0)) == 0.0


# ----------------------------------------------------------------- ranking
def test_top_k_brute_force(orc):
    """Top-k against a stable sort by (-variance, channel)."""
    r = _rng(4)
    for n_hi in (0, 16, 32, 64, 128):
        for trial in range(20):
            var = r.standard_normal(128).astype(np.float32)
            if trial % 3 == 0:
                var = np.round(var, 1).astype(np.float32)   # many ties
            order = np.lexsort((np.arange(128), -var.astype(np.float64)))
            want = np.zeros(128, bool)
            want[order[:n_hi]] = True
            assert (orc.top_k(var, n_hi) == want).all()


def test_top_k_ties_go_to_lower_index(orc):
    var = np.ones(128, np.float32)
    got = orc.top_k(var, 32)
    assert got[:32].all() and not got[32:].any()
    var = np.zeros(128, np.float32)
    var[5] = -0.0
    assert orc.top_k(var, 1)[0] and not orc.top_k(var, 1)[5]


def test_planted_outlier_channels_are_boosted(orc):
    """VeloxQuant-MLX docs, Evidence: high-variance channels correctly identified."""
    r = _rng(5)
    planted = np.sort(r.choice(128, 32, replace=False))
    scale = np.ones(128)
    scale[planted] = 10.0
    xk = _bf16(r.standard_normal((32, 128)) * scale)
    xv = _bf16(r.standard_normal((32, 128)))
    blob, st = orc.quantize_page_f32(xk, xv, 32)
    assert st == 0
    assert (orc.page_channels(blob, 32) == planted).all()


# ----------------------------------------------------------------- quantizer
def np_step(s):
    """Stored step for exact steps s >= 0 (float32 array): s rounded up to 7
    significant bits (numpy frexp / ceil / ldexp in float64), then up to the
    next fp16 value if it falls between two (only below the fp16 normal
    range).  Returned as float32 values."""
    s = np.asarray(s, np.float32).astype(np.float64)
    m, e = np.frexp(s)
    v = np.ldexp(np.ceil(np.ldexp(m, 7)), e - 7)
    h = v.astype(np.float16)
    h = np.where(h.astype(np.float64) < v, np.nextafter(h, np.float16(np.inf)), h)
    return h.astype(np.float32)


def test_step_rule(orc):
    """The stored step: the smallest fp16 value >= s with at most 7 significant
    bits.  Checked against numpy on random steps over the fp16 range, powers of
    two, values just above and below 7-bit boundaries, and fp16 subnormals."""
    r = _rng(3)
    s = (r.random(3000) * 10.0 ** r.integers(-9, 5, 3000)).astype(np.float32)
    edge = np.float32(1.0 + 2.0 ** -6)
    s = np.concatenate([s, np.float32(2.0) ** np.arange(-24, 15, dtype=np.float32),
                        [edge, np.nextafter(edge, np.float32(0)), np.nextafter(edge, np.float32(9)),
                         np.float32(3 * 2.0 ** -20), np.float32(1e-7), np.float32(0.0)]]).astype(np.float32)
    want = np_step(s)
    for x, w in zip(s, want):
        got = orc.f16_bits_to_f32(orc.step_f16(float(x)))
        assert got == w, (float(x), got, float(w))
        assert got >= x
        if x >= 2.0 ** -14:   # normal fp16: at most 7 significant bits, within 2^-6 above s
            assert (int(np.float16(got).view(np.uint16)) & 0xF) == 0
            assert got <= x * (1 + 2.0 ** -6)


def _np_uniform_quant(x, levels):
    """Per-channel asymmetric min/max quantizer over tokens (KIVI-style, fp16
    minimum, step np_step(s) (a boosted 4-bit channel stores np_step(4 s) and
    uses a quarter of it), codes rint((x - M) * (1/u)) in fp32, clamp): the
    textbook special case."""
    x = x.astype(np.float32)
    mn, mx = x.min(0), x.max(0)
    M = mn.astype(np.float16).astype(np.float32)
    s = ((mx - mn).astype(np.float32) / np.float32(levels)).astype(np.float32)
    if levels == 15:
        u = np_step(s * np.float32(4)) * np.float32(0.25)
    else:
        u = np_step(s)
    with np.errstate(divide="ignore", invalid="ignore"):
        # nearest integer to (x - M) times the reciprocal of the step, each rounded to fp32
        ru = np.where(u == 0, np.float32(0), np.float32(1) / np.where(u == 0, np.float32(1), u))
        code = np.clip(np.rint((x - M).astype(np.float32) * ru.astype(np.float32)), 0, levels)
    code = np.where(u == 0, 0, code)
    return M.astype(np.float64) + u.astype(np.float64) * code, code.astype(np.int64)


def _kv(seed, scale=None):
    r = _rng(seed)
    sig = np.exp(r.standard_normal(128)) if scale is None else scale
    return _bf16(r.standard_normal((32, 128)) * sig), _bf16(r.standard_normal((32, 128)))


def test_hf0_equals_uniform_2bit(orc):
    """hi_fraction = 0 is uniform 2-bit per-channel quantization (KIVI column of
    the comparison table)."""
    for seed in range(10):
        xk, xv = _kv(seed)
        blob, st = orc.quantize_page_f32(xk, xv, 0)
        kh, _, st2 = orc.dequant_page(blob, 0)
        want, _ = _np_uniform_quant(xk, 3)
        assert st == 0 and st2 == 0
        assert (kh == want).all()


def _np_uniform_4bit(x):
    """Textbook per-channel 4-bit asymmetric min/max quantizer that stores its own
    step: fp16 minimum, step u4 = np_step((max - min) / 15), codes
    clamp(rint((x - M) * (1/u4)), 0, 15) in fp32.  Returns (dequantized, the
    exact step s4)."""
    x = x.astype(np.float32)
    mn, mx = x.min(0), x.max(0)
    M = mn.astype(np.float16).astype(np.float32)
    s4 = ((mx - mn).astype(np.float32) / np.float32(15)).astype(np.float32)
    u4 = np_step(s4)
    with np.errstate(divide="ignore", invalid="ignore"):
        ru = np.where(u4 == 0, np.float32(0), np.float32(1) / np.where(u4 == 0, np.float32(1), u4))
        code = np.clip(np.rint((x - M).astype(np.float32) * ru.astype(np.float32)), 0, 15)
    code = np.where(u4 == 0, 0, code)
    return M.astype(np.float64) + u4.astype(np.float64) * code, s4


def test_hf1_equals_uniform_4bit(orc):
    """hi_fraction = 1 is uniform 4-bit per-channel quantization.  Kitty stores a
    boosted channel's high-plane step as the step of 4*s4 and decodes the 4-bit
    code with a quarter of it; an independent 4-bit quantizer stores the step of
    s4.  The two agree whenever s4 is a normal half (s4 >= 2^-14: scaling by a
    power of two commutes with both roundings there), so the decoded pages are
    identical on those channels.  Channels whose s4 lies below the fp16 normal
    range are excluded from the identity (there the fp16 grid is coarser
    relative to s4 than to 4*s4) and held to the quantizer's error bound
    instead; the last seeds plant such channels."""
    tiny_seen = 0
    for seed in range(12):
        xk, xv = _kv(seed)
        if seed >= 10:   # channels whose range is a few fp16 subnormal steps
            r = _rng(100 + seed)
            cols = r.choice(128, 16, replace=False)
            xk[:, cols] = _bf16(r.standard_normal((32, 16)) * 2.0 ** -14)
        blob, st = orc.quantize_page_f32(xk, xv, 128)
        kh, _, st2 = orc.dequant_page(blob, 128)
        assert st == 0 and st2 == 0
        want, s4 = _np_uniform_4bit(xk)
        normal = s4 >= np.float32(2.0 ** -14)
        assert (kh[:, normal] == want[:, normal]).all(), seed
        tiny = ~normal
        tiny_seen += int(tiny.sum())
        if tiny.any():
            x = xk[:, tiny].astype(np.float64)
            rng_ = x.max(0) - x.min(0)
            # within half a step: Kitty's step is S/4 with S at most 2^-6 above
            # 4*s4 and then at most 2^-24 (one fp16 subnormal ulp) above that;
            # plus the fp16 rounding of the minimum (half an ulp, 2^-25)
            bound = (rng_ / 15 * (1 + 2.0 ** -6) + 2.0 ** -26) / 2 + 2.0 ** -25
            assert (np.abs(kh[:, tiny] - x) <= bound[None, :] + 1e-12).all(), seed
    assert tiny_seen >= 16


def test_halfway_values_take_a_neighbouring_level(orc):
    """Values exactly halfway between two quantization levels, at steps 3*2^-m
    that are not powers of two (1/u is then inexact), for 3 levels (2-bit
    channels and Value groups), 15 (4-bit boosted channels of the (4, 2)
    configuration and 4-bit channels of (8, 4)) and 255 (8-bit boosted channels
    of (8, 4)): each decodes to one of its two neighbouring levels, the group
    ends decode exactly, and equal values get equal codes.  The planted columns
    have exact minima and steps, so the levels are minimum + step * k."""
    from tests.edge_inputs import half_way_column
    r = _rng(21)
    for lo_bit, n_hi, lv in ((2, 0, (3, 15)), (2, 128, (3, 15)), (4, 0, (15, 255)),
                             (4, 128, (15, 255))):
        levels = lv[1] if n_hi else lv[0]
        xk = np.zeros((32, 128))
        steps_k = np.zeros(128)
        for c in range(128):
            m, a = int(r.integers(2, 6)), int(r.integers(0, 3))
            xk[:, c] = half_way_column(levels, m, a)[r.permutation(32)]
            steps_k[c] = 3.0 * 2.0 ** -m
        xv = np.zeros((32, 128))
        steps_v = np.zeros((32, 4))
        for t in range(32):
            for G in range(4):
                m, a = int(r.integers(2, 6)), int(r.integers(0, 3))
                xv[t, 32 * G:32 * G + 32] = half_way_column(3, m, a)[r.permutation(32)]
                steps_v[t, G] = 3.0 * 2.0 ** -m
        assert (_bf16(xk) == xk).all() and (_bf16(xv) == xv).all()
        blob, st = orc.quantize_page_f32(xk, xv, n_hi, lo_bit=lo_bit)
        kh, vh, st2 = orc.dequant_page(blob, n_hi, lo_bit=lo_bit)
        assert st == 0 and st2 == 0
        groups = [(xk[:, c], kh[:, c], steps_k[c]) for c in range(128)]
        groups += [(xv[t, 32 * G:32 * G + 32], vh[t, 32 * G:32 * G + 32], steps_v[t, G])
                   for t in range(32) for G in range(4)]
        for x, xh, u in groups:
            mn = x.min()
            q = (x - mn) / u                      # exact: k + 1/2, or 0 / levels at the ends
            lo_, hi_ = mn + u * np.floor(q), mn + u * np.ceil(q)
            assert ((xh == lo_) | (xh == hi_)).all(), (lo_bit, n_hi)
            ends = (q == np.floor(q))
            assert (xh[ends] == x[ends]).all()
            for v in np.unique(x):
                assert len(set(xh[x == v].tolist())) == 1


def test_equal_variances_at_the_cut_go_to_lower_channels(orc):
    """Channels with equal variance straddling the n_hi cut (columns x or -x of
    one shared column): the boosted set is every larger-variance channel plus
    the lowest-indexed tied channels (brute force over the planted roles)."""
    from tests.edge_inputs import tie_columns, tie_tile
    r = _rng(22)
    for n_distinct, n_tied, n_hi in ((0, 40, 32), (20, 30, 32), (5, 20, 16), (10, 60, 64)):
        for lo_bit in (2, 4):
            d, t, sg = tie_columns(r, n_distinct, n_tied)
            xk = synth.from_bits(tie_tile(r, d, t, sg, synth.BF16), synth.BF16)
            xv = _bf16(r.standard_normal((32, 128)))
            blob, st = orc.quantize_page_f32(xk, xv, n_hi, lo_bit=lo_bit)
            assert st == 0
            want = np.sort(np.concatenate([d, t[:n_hi - n_distinct]]))
            assert (orc.page_channels(blob, n_hi, lo_bit=lo_bit) == want).all()


def _planes(blob, n_hi):
    base = np.zeros((32, 128), np.int64)
    for c in range(128):
        for t in range(32):
            w, b = orc_pos_cache("k", c, t, 8)
            base[t, c] = (int.from_bytes(bytes(blob[4 * w:4 * w + 4]), "little") >> b) & 3
    extra = np.zeros((32, n_hi), np.int64)
    off = 1024
    for j in range(n_hi):
        for t in range(32):
            w, b = orc_pos_cache("k", j, t, n_hi // 16)
            extra[t, j] = (int.from_bytes(bytes(blob[off + 4 * w:off + 4 * w + 4]), "little") >> b) & 3
    return base, extra


_POS = {}


def orc_pos_cache(kind, a, b, wpl=8):
    key = (kind, a, b, wpl)
    if key not in _POS:
        import oracle
        _POS[key] = oracle.key_pos(a, b, wpl) if kind == "k" else oracle.val_pos(a, b)
    return _POS[key]


def test_planes_recombine_to_4bit_code(orc):
    """Paper abstract: a mixed-precision Key page is two uniform 2-bit tensors.
    For every boosted element 4*hi + lo equals the 4-bit code."""
    xk, xv = _kv(11)
    blob, _ = orc.quantize_page_f32(xk, xv, 32)
    base, extra = _planes(blob, 32)
    kch = orc.page_channels(blob, 32).astype(np.int64)
    assert (np.diff(kch) > 0).all()
    _, code4 = _np_uniform_quant(xk, 15)
    for j, c in enumerate(kch):
        assert (4 * base[:, c] + extra[:, j] == code4[:, c]).all()
    normal = np.setdiff1d(np.arange(128), kch)
    _, code2 = _np_uniform_quant(xk, 3)
    assert (base[:, normal] == code2[:, normal]).all()


def test_plane_maps_are_bijections(orc):
    seen = set()
    for c in range(128):
        for t in range(32):
            seen.add(orc.key_pos(c, t, 8))
    assert len(seen) == 4096 and {w for w, _ in seen} == set(range(256))
    assert {b for _, b in seen} == set(range(0, 32, 2))
    seen = set()
    for t in range(32):
        for c in range(128):
            seen.add(orc.val_pos(t, c))
    assert len(seen) == 4096 and {w for w, _ in seen} == set(range(256))
    for nh in (16, 32, 64):
        seen = {orc.key_pos(j, t, nh // 16) for j in range(nh) for t in range(32)}
        assert len(seen) == nh * 32 and max(w for w, _ in seen) == nh * 2 - 1
    assert sorted(orc.meta_pos("km", c) for c in range(128)) == list(range(128))
    assert sorted(orc.meta_pos("vmeta", g, t) for g in range(4) for t in range(32)) == list(range(128))
    assert sorted(orc.meta_pos("kch", j) for j in range(64)) == list(range(64))


def test_closed_forms_exact_reconstruction(orc):
    """Constant channels decode exactly (step 0, codes 0); values on a power-of-two
    grid {0..3}*delta (2-bit) and {0..15}*delta (boosted) decode exactly; codes are
    monotone in the input."""
    r = _rng(12)
    xk = np.zeros((32, 128), np.float32)
    for c in range(128):
        delta = 2.0 ** int(r.integers(2, 5)) if c < 32 else 2.0 ** int(r.integers(-6, 2))
        off = float(r.integers(-8, 8))
        if c < 32:       # high variance: will be boosted, 16-level grid
            xk[:, c] = off + delta * 4 * r.integers(0, 16, 32)
            xk[0, c], xk[1, c] = off, off + delta * 4 * 15
        elif c < 64:     # constant
            xk[:, c] = off + delta
        else:
            xk[:, c] = off + delta * r.integers(0, 4, 32) * 0.25
            xk[0, c], xk[1, c] = off, off + delta * 0.75
    # Values: every (token, group of 32 channels) has its own offset and
    # power-of-two step, so only the right group's metadata decodes them exactly
    xv = np.zeros((32, 128), np.float32)
    for t in range(32):
        for G in range(4):
            q = r.integers(0, 4, 32)
            q[0], q[1] = 0, 3
            xv[t, 32 * G:32 * G + 32] = float(r.integers(-8, 8)) + 2.0 ** int(r.integers(-4, 3)) * q
    blob, st = orc.quantize_page_f32(xk, xv, 32)
    kh, vh, _ = orc.dequant_page(blob, 32)
    assert st == 0
    assert (kh == xk.astype(np.float64)).all()
    assert (vh == xv.astype(np.float64)).all()
    xk2, xv2 = _kv(13)
    blob, _ = orc.quantize_page_f32(xk2, xv2, 32)
    base, extra = _planes(blob, 32)
    kch = orc.page_channels(blob, 32)
    code = base.copy()
    for j, c in enumerate(kch):
        code[:, c] = 4 * base[:, c] + extra[:, j]
    for c in range(128):
        o = np.argsort(xk2[:, c], kind="stable")
        assert (np.diff(code[o, c]) >= 0).all()


def test_signed_zero_min_max_is_order_free(orc):
    """Of two zeros, -0 is the minimum and +0 the maximum (IEEE 754-2019
    minimum/maximum; the pages say only "min/max"): a Key channel or Value group
    whose minimum is a zero stores M = -0 (0x8000) whenever a -0 is present, in
    any token order, and +0 (0x0000) when none is; a group of zeros has step +0."""
    xk, xv = _kv(40)
    r = _rng(41)
    z = np.where(r.permutation(np.r_[np.zeros(16), np.ones(16)]) == 1,
                 np.float32(-0.0), np.float32(0.0)).astype(np.float32)
    xk[:, 3] = z                                   # zeros, random signs
    xk[:, 4] = z[::-1]                             # the same, reversed order
    xk[:, 5] = 0.0                                 # +0 only
    xk[:, 6] = np.abs(xk[:, 6]) + 1.0
    xk[7, 6], xk[19, 6] = 0.0, -0.0                # minimum a zero, both signs
    xv[0, 0:32] = z
    xv[1, 32:64] = z[::-1]
    xv[2, 64:96] = 0.0
    blob, st = orc.quantize_page_f32(xk, xv, 32)
    assert st == 0
    lay = dict(ks=1280, km=1536, vs=2848, vm=3104)   # n_hi = 32, 2-bit planes
    u16 = lambda off, i: int(blob[off + 2 * i]) | (int(blob[off + 2 * i + 1]) << 8)
    km = lambda c: u16(lay["km"], orc.meta_pos("km", c))
    assert km(3) == 0x8000 and km(4) == 0x8000 and km(6) == 0x8000
    assert km(5) == 0x0000
    assert u16(lay["ks"], 3) == u16(lay["ks"], 4) == u16(lay["ks"], 5) == 0x0000
    vm = lambda g, t: u16(lay["vm"], orc.meta_pos("vmeta", g, t))
    vs = lambda g, t: u16(lay["vs"], orc.meta_pos("vmeta", g, t))
    assert vm(0, 0) == 0x8000 and vm(1, 1) == 0x8000 and vm(2, 2) == 0x0000
    assert vs(0, 0) == vs(1, 1) == vs(2, 2) == 0x0000
    kh, vh, _ = orc.dequant_page(blob, 32)
    assert (kh[:, 3:6] == 0).all() and (vh[0, 0:32] == 0).all()


def test_reconstruction_error_bound(orc):
    """|x - xhat| <= step/2 inside the stored range; clamped values lose at most the
    fp16 rounding of the minimum / of the top of the range."""
    for seed in range(20, 30):
        xk, xv = _kv(seed)
        blob, _ = orc.quantize_page_f32(xk, xv, 32)
        kh, vh, _ = orc.dequant_page(blob, 32)
        kch = set(orc.page_channels(blob, 32).tolist())
        for x, xh, groups in ((xk, kh, [(slice(None), c) for c in range(128)]),
                              (xv, vh, [(t, slice(32 * g, 32 * g + 32)) for t in range(32) for g in range(4)])):
            for sel in groups:
                a = x[sel].astype(np.float64)
                ah = xh[sel]
                mn, mx = a.min(), a.max()
                M = float(np.float32(mn).astype(np.float16))
                boosted = x is xk and sel[1] in kch
                L = 15 if boosted else 3
                s = np.float32(np.float32(mx - mn) / np.float32(L))
                u = float(np_step(4 * s)) / 4 if boosted else float(np_step(s))
                bound = max(u / 2 * (1 + 1e-6), M - mn, mx - (M + L * u)) + 1e-6 * abs(a).max()
                assert np.abs(ah - a).max() <= bound + 1e-12


def test_boost_lowers_error(orc):
    """VeloxQuant-MLX docs, Evidence: mixed precision beats uniform 2-bit on
    high-variance data, and boosted channels show a lower normalised error than
    2-bit channels."""
    tot_k = tot_u = 0.0
    hi_err, lo_err = [], []
    for seed in range(40, 60):
        xk, xv = _kv(seed)
        blob, _ = orc.quantize_page_f32(xk, xv, 32)
        kh, _, _ = orc.dequant_page(blob, 32)
        uni, _ = _np_uniform_quant(xk, 3)
        e_k = (kh - xk) ** 2
        e_u = (uni - xk) ** 2
        # grid inclusion (j = 5k) up to the rounding of the two stored steps: each
        # is at most 2^-6 above its exact step, so grid point k moves by at most
        # 3 * 2^-6 * (max - min) / 3
        rng_ = xk.astype(np.float64).max(0) - xk.astype(np.float64).min(0)
        assert (np.abs(kh - xk) <= np.abs(uni - xk) + 2.0 ** -6 * rng_ + 1e-6).all()
        tot_k += e_k.sum()
        tot_u += e_u.sum()
        kch = orc.page_channels(blob, 32)
        var = xk.astype(np.float64).var(0) + 1e-30
        norm = e_k.mean(0) / var
        mask = np.zeros(128, bool)
        mask[kch] = True
        hi_err.append(norm[mask].mean())
        lo_err.append(norm[~mask].mean())
    assert tot_k < 0.5 * tot_u
    assert np.mean(hi_err) < 0.2 * np.mean(lo_err)


# ----------------------------------------------------------------- running statistics
def test_running_one_page_equals_page_mode(orc):
    for seed in range(5):
        xk, xv = _kv(100 + seed)
        a, _ = orc.quantize_page_f32(xk, xv, 32)
        rs, rq, rc = np.zeros(128, np.float32), np.zeros(128, np.float32), np.zeros(1, np.int32)
        b, _ = orc.quantize_page_f32(xk, xv, 32, (rs, rq, rc))
        assert (a == b).all() and rc[0] == 32


def test_running_variance_tracks_all_tokens(orc):
    """VeloxQuant-MLX docs, Decode phase step 2: the running estimate follows the
    variance over every token seen so far."""
    r = _rng(7)
    rs, rq, rc = np.zeros(128, np.float32), np.zeros(128, np.float32), np.zeros(1, np.int32)
    seen = []
    sig = np.exp(r.standard_normal(128))
    for p in range(12):
        xk = _bf16(r.standard_normal((32, 128)) * sig + 0.5)
        orc.quantize_page_f32(xk, xk, 32, (rs, rq, rc))
        seen.append(xk.astype(np.float64))
        allx = np.concatenate(seen)
        for c in range(0, 128, 9):
            v = float(orc.variance(rs[c], rq[c], float(rc[0])))
            assert abs(v - allx[:, c].var()) <= 1e-5 * (allx[:, c] ** 2).mean()


def _empty_state(B, Hkv, max_pages, pool_pages, n_hi):
    return dict(tail_k=np.zeros((B, Hkv, 32, 128), np.uint16), tail_v=np.zeros((B, Hkv, 32, 128), np.uint16),
                tail_len=np.zeros(B, np.int32), run_sum=np.zeros((B, Hkv, 128), np.float32),
                run_sumsq=np.zeros((B, Hkv, 128), np.float32), run_count=np.zeros((B, Hkv), np.int32),
                block_table=np.full((B, max_pages), -1, np.int32), num_pages=np.zeros(B, np.int32),
                pool=np.zeros(pool_pages * Hkv * 3072 + pool_pages * Hkv * 9 * n_hi, np.uint8))


def test_append_equals_bulk_running(orc):
    """Appending tokens one at a time (flushing every 32nd) writes the same bytes
    as quantizing the same pages in bulk in running mode."""
    B, Hkv, n_hi, npg = 2, 2, 32, 3
    r = _rng(8)
    toks_k = synth.to_bits(r.standard_normal((B, npg * 32, Hkv, 128)) * np.exp(r.standard_normal(128)), synth.BF16)
    toks_v = synth.to_bits(r.standard_normal((B, npg * 32, Hkv, 128)), synth.BF16)
    ids = np.array([[4, 1, 5], [0, 3, 2]], np.int32)
    st = _empty_state(B, Hkv, npg, B * npg, n_hi)
    for t in range(npg * 32):
        fl = np.where((st["tail_len"] + 1) == 32, ids[np.arange(B), st["num_pages"]], -1).astype(np.int32)
        s = orc.append_token(Hkv, n_hi, 1, synth.BF16, toks_k[:, t], toks_v[:, t], st["tail_k"], st["tail_v"],
                             st["tail_len"], st["run_sum"], st["run_sumsq"], st["run_count"], fl,
                             st["block_table"], npg, st["num_pages"], st["pool"], B * npg)
        assert s == 0
    assert (st["num_pages"] == npg).all() and (st["tail_len"] == 0).all()
    assert (st["block_table"] == ids).all()
    pool2 = np.zeros_like(st["pool"])
    rs = np.zeros((B, Hkv, 128), np.float32)
    rq = np.zeros_like(rs)
    rc = np.zeros((B, Hkv), np.int32)
    k = toks_k.reshape(B * npg * 32, Hkv, 128)
    v = toks_v.reshape(B * npg * 32, Hkv, 128)
    s = orc.quantize_pages(Hkv, n_hi, 1, synth.BF16, k, v, ids.reshape(-1), pool2, B * npg,
                           seq_of_page=np.repeat(np.arange(B), npg), n_seqs=B, run_sum=rs,
                           run_sumsq=rq, run_count=rc)
    assert s == 0
    assert (pool2 == st["pool"]).all()
    assert (rs == st["run_sum"]).all() and (rq == st["run_sumsq"]).all() and (rc == st["run_count"]).all()


def test_append_status_codes(orc):
    B, Hkv, n_hi = 1, 1, 32
    st = _empty_state(B, Hkv, 1, 1, n_hi)
    kn = np.zeros((1, 1, 128), np.uint16)

    def app(fl):
        return orc.append_token(Hkv, n_hi, 1, synth.BF16, kn, kn, st["tail_k"], st["tail_v"],
                                st["tail_len"], st["run_sum"], st["run_sumsq"], st["run_count"],
                                np.array([fl], np.int32), st["block_table"], 1, st["num_pages"],
                                st["pool"], 1)
    assert app(0) == orc.ST["BAD_FLUSH"] and st["tail_len"][0] == 1
    for _ in range(30):
        assert app(-1) == 0
    assert app(-1) == 0 and st["tail_len"][0] == 32
    assert app(-1) == orc.ST["TAIL_FULL"]


# ----------------------------------------------------------------- attention
def _build(orc, w, seed=0):
    inp = synth.host_inputs(w, seed)
    blob = orc.page_bytes(w.n_hi)
    pool = np.zeros(inp["pool_pages"] * w.Hkv * blob, np.uint8)
    st = orc.quantize_pages(w.Hkv, w.n_hi, 0, w.dtype, inp["k"], inp["v"], inp["page_ids"], pool,
                            inp["pool_pages"])
    assert st == 0
    return inp, pool


def _np_attention(orc, w, inp, pool, sm):
    """Softmax attention with numpy over the oracle's dequantized pages."""
    blob = orc.page_bytes(w.n_hi)
    out = np.zeros((w.B, w.Hq, 128))
    for b in range(w.B):
        for kvh in range(w.Hkv):
            ks, vs = [], []
            for p in range(inp["num_pages"][b]):
                pid = inp["block_table"][b, p]
                off = (pid * w.Hkv + kvh) * blob
                kh, vh, _ = orc.dequant_page(pool[off:off + blob], w.n_hi)
                ks.append(kh)
                vs.append(vh)
            tl = inp["tail_len"][b]
            ks.append(synth.from_bits(inp["tail_k"][b, kvh, :tl], w.dtype).astype(np.float64))
            vs.append(synth.from_bits(inp["tail_v"][b, kvh, :tl], w.dtype).astype(np.float64))
            K, V = np.concatenate(ks), np.concatenate(vs)
            for h in range(w.g):
                q = synth.from_bits(inp["q"][b, kvh * w.g + h], w.dtype).astype(np.float64)
                if len(K) == 0:
                    continue
                s = sm * (K @ q)
                p_ = np.exp(s - s.max())
                out[b, kvh * w.g + h] = (p_ / p_.sum()) @ V
    return out


@pytest.mark.parametrize("name", ["tiny", "small_gqa"])
def test_attention_against_numpy(orc, name):
    w = synth.workload(name)
    inp, pool = _build(orc, w)
    sm = float(np.float32(1 / math.sqrt(128)))   # the API takes the scale as fp32
    out, st = orc.decode_attention(w.Hkv, w.Hq, w.n_hi, w.dtype, inp["q"], pool, inp["pool_pages"],
                                   inp["block_table"], inp["num_pages"], inp["tail_k"], inp["tail_v"],
                                   inp["tail_len"], sm)
    want = _np_attention(orc, w, inp, pool, sm)
    assert st == 0
    assert np.abs(out - want).max() <= 1e-12 * max(1.0, np.abs(want).max())
    out2, _ = orc.decode_attention(w.Hkv, w.Hq, w.n_hi, w.dtype, inp["q"], pool, inp["pool_pages"],
                                   inp["block_table"], inp["num_pages"], inp["tail_k"], inp["tail_v"],
                                   inp["tail_len"], sm)
    assert (out == out2).all()


def test_attention_closed_forms(orc):
    """One token: o = v.  Identical keys: o = mean of v.  Empty: o = 0, EMPTY."""
    Hkv = Hq = 1
    r = _rng(9)
    q = synth.to_bits(r.standard_normal((1, 1, 128)), synth.BF16)
    tk = np.zeros((1, 1, 32, 128), np.uint16)
    tv = synth.to_bits(r.standard_normal((1, 1, 32, 128)), synth.BF16)
    tk[:] = synth.to_bits(r.standard_normal(128), synth.BF16)
    bt = np.zeros((1, 1), np.int32)
    pool = np.zeros(3360, np.uint8)
    for n in (1, 7, 32):
        out, st = orc.decode_attention(Hkv, Hq, 32, synth.BF16, q, pool, 1, bt, np.array([0], np.int32),
                                       tk, tv, np.array([n], np.int32), 0.1)
        want = synth.from_bits(tv[0, 0, :n], synth.BF16).astype(np.float64).mean(0)
        assert st == 0 and np.abs(out[0, 0] - want).max() <= 1e-12
    out, st = orc.decode_attention(Hkv, Hq, 32, synth.BF16, q, pool, 1, bt, np.array([0], np.int32),
                                   tk, tv, np.array([0], np.int32), 0.1)
    assert st == orc.ST["EMPTY"] and (out == 0).all()
    # one dominant score: key parallel to q with a large norm
    tk2 = synth.to_bits(np.zeros((1, 1, 32, 128)), synth.BF16)
    qf = synth.from_bits(q[0, 0], synth.BF16)
    tk2[0, 0, 3] = synth.to_bits(qf * 8, synth.BF16)
    out, _ = orc.decode_attention(Hkv, Hq, 32, synth.BF16, q, pool, 1, bt, np.array([0], np.int32),
                                  tk2, tv, np.array([5], np.int32), 1.0)
    assert np.abs(out[0, 0] - synth.from_bits(tv[0, 0, 3], synth.BF16)).max() < 1e-9


def test_attention_bad_page_id(orc):
    w = synth.workload("tiny")
    inp, pool = _build(orc, w)
    bt = inp["block_table"].copy()
    bt[0, 2] = 1000
    _, st = orc.decode_attention(w.Hkv, w.Hq, w.n_hi, w.dtype, inp["q"], pool, inp["pool_pages"], bt,
                                 inp["num_pages"], inp["tail_k"], inp["tail_v"], inp["tail_len"], 0.1)
    assert st == orc.ST["BAD_PAGE"]


def test_quantize_range_status(orc):
    xk, xv = _kv(3)
    xk[4, 7] = 70000.0
    _, st = orc.quantize_page_f32(xk, xv, 32)
    assert st == orc.ST["RANGE"]
    xk[4, 7] = np.nan
    _, st = orc.quantize_page_f32(xk, xv, 32)
    assert st == orc.ST["NONFINITE"]


# ----------------------------------------------------------------- sequence-wide ranking
def _seq_pages(seed, npg, offsets=None):
    r = _rng(seed)
    sig = np.exp(r.standard_normal(128))
    k = r.standard_normal((npg * 32, 1, 128)) * sig
    if offsets is not None:
        k += offsets[:, None, :].repeat(32, axis=0)
    return (synth.to_bits(k, synth.BF16), synth.to_bits(r.standard_normal((npg * 32, 1, 128)), synth.BF16))


def _quant(orc, mode, k, v, npg):
    pool = np.zeros(npg * orc.page_bytes(32), np.uint8)
    rs = np.zeros((1, 1, 128), np.float32)
    rq = np.zeros_like(rs)
    rc = np.zeros((1, 1), np.int32)
    st = orc.quantize_pages(1, 32, mode, synth.BF16, k, v, np.arange(npg), pool, npg,
                            seq_of_page=np.zeros(npg, np.int32), n_seqs=1, run_sum=rs, run_sumsq=rq,
                            run_count=rc)
    assert st == 0
    return pool, (rs, rq, rc)


def test_sequence_mode_one_page_equals_other_modes(orc):
    k, v = _seq_pages(30, 1)
    a, _ = _quant(orc, 0, k, v, 1)
    b, _ = _quant(orc, 1, k, v, 1)
    c, _ = _quant(orc, 2, k, v, 1)
    assert (a == b).all() and (a == c).all()


def test_sequence_mode_ranks_over_the_whole_prompt(orc):
    """VeloxQuant-MLX docs, Prefill phase step 1: variance across the sequence axis.
    Channels that are constant inside each page but jump between pages have ~0
    variance per page and a large variance over the sequence: the sequence mode
    boosts exactly them, on every page; the page mode does not."""
    r = _rng(31)
    npg = 8
    planted = np.sort(r.choice(128, 32, replace=False))
    off = np.zeros((npg, 128))
    off[:, planted] = r.standard_normal((npg, 32)) * 50.0
    k, v = _seq_pages(32, npg, off)
    k_view = synth.from_bits(k, synth.BF16)
    k_view[:, :, planted] = synth.from_bits(synth.to_bits(off[:, None, planted].repeat(32, 0).reshape(-1, 1, 32),
                                                          synth.BF16), synth.BF16)
    k = synth.to_bits(k_view, synth.BF16)
    pool, (rs, rq, rc) = _quant(orc, 2, k, v, npg)
    blob = orc.page_bytes(32)
    for p in range(npg):
        assert (orc.page_channels(pool[p * blob:(p + 1) * blob], 32) == planted).all()
    page_pool, _ = _quant(orc, 0, k, v, npg)
    assert not all((orc.page_channels(page_pool[p * blob:(p + 1) * blob], 32) == planted).all()
                   for p in range(npg))
    run_pool, (rs1, rq1, rc1) = _quant(orc, 1, k, v, npg)
    assert (rs == rs1).all() and (rq == rq1).all() and (rc == rc1).all() and rc[0, 0] == 32 * npg


# ----------------------------------------------------------------- 16-bit paged baseline
def test_f16kv_attention_against_numpy(orc):
    """The unquantized 16-bit paged layout (the comparison layout of the paper's
    same-budget claims, Abstract): the oracle's fp64 attention over pages in
    block-table order equals numpy's softmax attention over the token rows,
    with ragged lengths (a partial last page), grouped heads (query head h
    reads kv head h / g), an empty sequence (0 and EMPTY) and a bad page id."""
    r = _rng(31)
    Hkv, Hq, D, P = 2, 6, 128, 32
    lens = np.array([70, 1, 0, 64], np.int32)
    max_pages = 3
    pool_pages = 12
    for dt in (synth.BF16, synth.F16):
        pool = synth.to_bits(r.standard_normal((pool_pages, Hkv, 2, P, D)), dt)
        ids = r.permutation(pool_pages)[:len(lens) * max_pages].reshape(len(lens), max_pages).astype(np.int32)
        q = synth.to_bits(r.standard_normal((len(lens), Hq, D)), dt)
        scale = float(np.float32(1 / np.sqrt(D)))
        out, st = orc.decode_f16kv(Hkv, Hq, dt, q, pool, pool_pages, ids, lens, scale)
        assert st == orc.ST["EMPTY"]
        kv = synth.from_bits(pool, dt).astype(np.float64)
        qf = synth.from_bits(q, dt).astype(np.float64)
        for b, L in enumerate(lens):
            for hq in range(Hq):
                h = hq // (Hq // Hkv)
                if L == 0:
                    assert (out[b, hq] == 0).all()
                    continue
                t = np.arange(L)
                K = kv[ids[b, t // P], h, 0, t % P]
                V = kv[ids[b, t // P], h, 1, t % P]
                s = K @ qf[b, hq] * scale
                w = np.exp(s - s.max())
                ref = (w / w.sum()) @ V
                assert np.abs(out[b, hq] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())
        bad = ids.copy()
        bad[0, 1] = pool_pages + 3
        _, st = orc.decode_f16kv(Hkv, Hq, dt, q, pool, pool_pages, bad, lens, scale)
        assert st == orc.ST["BAD_PAGE"]
