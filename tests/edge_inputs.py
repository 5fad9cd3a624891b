"""Planted inputs for the quantizer's edge cases, shared by the oracle pins (CPU)
and the GPU parity tests.  They only place values; none of the method's
arithmetic is here.

* Ranking ties: Key channels whose columns are x or -x of one shared column, so
  their sums of squares are equal and their sums equal up to sign: equal
  variances, in page, running and sequence statistics alike.
* Rounding ties: channels (and Value groups) whose values sit exactly halfway
  between two quantization levels, at steps 3 * 2^-m that are not powers of
  two, for 3, 15 and 255 levels.
"""

from __future__ import annotations

import numpy as np

from mixed_precision_bit_gb300 import synth

D, PAGE = 128, 32


def _bits(x, dtype):
    b = synth.to_bits(np.asarray(x, np.float64), dtype)
    back = synth.from_bits(b, dtype)
    assert (back == np.asarray(x, np.float64)).all(), "planted value not exact in the input dtype"
    return b


def tie_columns(rng, n_distinct, n_tied, n_other=None):
    """Channel roles of one Key tile: (distinct, tied, signs), channel index arrays.
    distinct: n_distinct channels with larger, distinct variances; tied: n_tied
    channels sharing one column up to sign (equal variances)."""
    perm = rng.permutation(D)
    distinct = np.sort(perm[:n_distinct])
    tied = np.sort(perm[n_distinct:n_distinct + n_tied])
    signs = rng.choice(np.array([-1.0, 1.0]), size=n_tied)
    return distinct, tied, signs


def tie_tile(rng, distinct, tied, signs, dtype):
    """One 32-token Key tile [32][128] (input-dtype bits): the distinct channels
    at scale 64 (each its own column), the tied ones +-x at scale 8, the rest at
    scale 1."""
    x = rng.standard_normal((PAGE, D))
    base = synth.from_bits(synth.to_bits(rng.standard_normal(PAGE) * 8.0, dtype), dtype)
    x[:, distinct] *= 64.0
    x[:, tied] = base[:, None] * signs[None, :]
    return synth.to_bits(x, dtype)


def plant_ties(inp, w, seed, n_distinct, n_tied):
    """Ranking ties in every (page, kv head) of inp["k"] (in place).  The tied
    channel set is fixed per (sequence, kv head), so running and sequence
    totals tie too; the shared column differs per page.  Returns the roles
    {(seq, head): (distinct, tied)}."""
    rng = np.random.default_rng(seed)
    roles = {}
    off = 0
    for b in range(w.B):
        for h in range(w.Hkv):
            roles[(b, h)] = tie_columns(rng, n_distinct, n_tied)
        for p in range(int(w.pages[b])):
            t0 = (off + p) * PAGE
            for h in range(w.Hkv):
                d, t, s = roles[(b, h)]
                inp["k"][t0:t0 + PAGE, h, :] = tie_tile(rng, d, t, s, w.dtype)
        off += int(w.pages[b])
    return {k: v[:2] for k, v in roles.items()}


def half_way_column(levels, m, a, boosted_w=None):
    """32 values of one channel (or Value group) whose quantizer step is
    u = 3 * 2^-m and whose quotients (x - minimum) / u are 0, levels and, for
    the other 30 values, exact halves k + 1/2.

    levels 3 or 15: minimum -a*u, maximum (levels - a)*u, so the range over
    levels is u exactly.  levels 255 (an 8-bit boosted code): minimum -2^-m,
    maximum 764 * 2^-m, range 765 * 2^-m = 255 * u.  Values are listed with
    the two ends first."""
    u = 3.0 * 2.0 ** -m
    if levels == 255:
        mn, mx = -(2.0 ** -m), 764.0 * 2.0 ** -m
        ks = np.arange(30) % 43              # 6k + 1 <= 253: exact in bf16
    else:
        mn, mx = -a * u, (levels - a) * u
        ks = np.arange(30) % levels
    vals = np.concatenate([[mn, mx], mn + (ks + 0.5) * u])
    return vals


def plant_half_way(inp, w, key_levels, boosted, seed, value_levels=3):
    """Rounding ties in every Key channel and Value group of every page
    (in place).  key_levels: (levels of a normal channel, levels of a boosted
    one); boosted: channel indices given the larger scale, so that a ranking
    of n_hi = len(boosted) boosts exactly them; value_levels: 3 (2-bit Values)
    or 15 (4-bit)."""
    rng = np.random.default_rng(seed)
    tot = int(w.pages.sum())
    is_b = np.zeros(D, bool)
    is_b[boosted] = True
    for p in range(tot):
        t0 = p * PAGE
        for h in range(w.Hkv):
            kt = np.zeros((PAGE, D))
            for c in range(D):
                lv = key_levels[1] if is_b[c] else key_levels[0]
                m = int(rng.integers(1, 3)) if is_b[c] else int(rng.integers(5, 8))
                col = half_way_column(lv, m, int(rng.integers(0, 3)))
                kt[:, c] = col[rng.permutation(PAGE)]
            inp["k"][t0:t0 + PAGE, h, :] = _bits(kt, w.dtype)
            vt = np.zeros((PAGE, D))
            for t in range(PAGE):
                for G in range(4):
                    col = half_way_column(value_levels, int(rng.integers(2, 7)),
                                          int(rng.integers(0, 3)))
                    vt[t, 32 * G:32 * G + 32] = col[rng.permutation(32)]
            inp["v"][t0:t0 + PAGE, h, :] = _bits(vt, w.dtype)
    return inp
