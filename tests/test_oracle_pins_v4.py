"""Pins of the oracle's 4-bit Value format (v_bit = 4, with 4-bit Key planes):
the uniform 4-bit KV cache that the Kitty paper's Abstract names as the
accuracy-preserving point ("4-bit KV quantization preserves accuracy"), here
per-channel 4-bit Keys (n_hi = 0 at lo_bit 4) and per-token 4-bit Value groups
of 32 channels, and Kitty (8, 4) Keys with 4-bit Values.

Each pin checks the oracle against an independent statement of the same fact:
the per-group quantizer written here from its textbook definition (applied to
Value groups), the nibble map enumerated by brute force, closed forms, the grid
inclusion that orders the 2-bit and 4-bit Value errors, and fp64 softmax
attention over the dequantized pages.
"""

import math

import numpy as np

from mixed_precision_bit_gb300 import synth
from tests.test_oracle_pins_84 import _np_quant


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16(x):
    return synth.from_bits(synth.to_bits(np.asarray(x, np.float32), synth.BF16), synth.BF16)


def _kv(seed):
    r = _rng(seed)
    sig = np.exp(r.standard_normal(128))
    return _bf16(r.standard_normal((32, 128)) * sig), _bf16(r.standard_normal((32, 128)) * 3)


def _groups(xv):
    """[32 tokens][128] -> [32 channels of a group][(token, group)]: the axis the
    per-group quantizer reduces over comes first."""
    return xv.reshape(32, 4, 32).transpose(2, 0, 1).reshape(32, 128)


def _ungroup(x):
    return x.reshape(32, 32, 4).transpose(1, 2, 0).reshape(32, 128)


def _np_value_quant(xv, levels):
    rec, code = _np_quant(_groups(xv), levels)
    return _ungroup(rec), _ungroup(code)


def test_page_bytes_v4(orc):
    """The Value plane doubles to 2048 B (4 bits x 32 x 128); everything else is
    the (8, 4) layout: 5120 + 17 * n_hi.  4-bit Values need 4-bit Key planes."""
    for nh in (0, 16, 32, 128):
        assert orc.page_bytes(nh, 4, 4) == 2048 + 16 * nh + 512 + nh + 2048 + 512
    assert orc.page_bytes(32, 2, 4) == -1 and orc.page_bytes(32, 4, 3) == -1


def test_value_nibble_map_is_a_bijection(orc):
    seen = {orc.val_pos4(t, c) for t in range(32) for c in range(128)}
    assert len(seen) == 4096
    assert {w for w, _ in seen} == set(range(512))
    assert {b for _, b in seen} == set(range(2, 32, 4))   # nibble starts, rotated by 2
    # fragment order: lane L = 4r + qq (words 16L..16L+15) holds channels with
    # c % 8 == r and tokens with (t % 8) // 2 == qq, and the 8 nibbles of a word
    # are one m16n8k16 A fragment: rows r, r + 8 of one 16-channel tile times
    # columns 2qq, 2qq + 1, 2qq + 8, 2qq + 9 of one 16-token tile
    words = {}
    for t in range(32):
        for c in range(128):
            wd, _ = orc.val_pos4(t, c)
            assert (wd // 16) // 4 == c % 8 and (wd // 16) % 4 == (t % 8) // 2
            words.setdefault(wd, set()).add((c // 16, t // 16))
    assert all(len(v) == 1 for v in words.values())


def _value_codes(orc, blob, n_hi):
    vbase = 2048 + 16 * n_hi + 512 + n_hi

    def nib(w, b):
        x = int.from_bytes(bytes(blob[vbase + 4 * w:vbase + 4 * w + 4]), "little")
        return ((x >> b) | (x << (32 - b))) & 15   # a nibble at bit 30 wraps to bit 0
    return np.array([[nib(*orc.val_pos4(t, c)) for c in range(128)] for t in range(32)])


def test_uniform_4bit_kv(orc):
    """n_hi = 0, lo_bit = 4, v_bit = 4: Keys decode as an independent per-channel
    4-bit quantizer, Values as an independent per-(token, group) 4-bit quantizer,
    and the Value codes sit in the plane where the nibble map says."""
    for seed in range(6):
        xk, xv = _kv(seed)
        blob, st = orc.quantize_page_f32(xk, xv, 0, lo_bit=4, v_bit=4)
        kh, vh, st2 = orc.dequant_page(blob, 0, lo_bit=4, v_bit=4)
        assert st == 0 and st2 == 0
        assert (kh == _np_quant(xk, 15)[0]).all()
        want, code = _np_value_quant(xv, 15)
        assert (vh == want).all()
        assert (_value_codes(orc, blob, 0) == code).all()


def test_kitty_84_with_4bit_values(orc):
    """n_hi = 32 at (8, 4) with v_bit = 4: the Key part of the blob is the same
    as with 2-bit Values; the Values are the 4-bit group quantizer's."""
    for seed in range(6, 10):
        xk, xv = _kv(seed)
        b2, _ = orc.quantize_page_f32(xk, xv, 32, lo_bit=4)
        b4, _ = orc.quantize_page_f32(xk, xv, 32, lo_bit=4, v_bit=4)
        vbase = 2048 + 16 * 32 + 512 + 32
        assert (b2[:vbase] == b4[:vbase]).all()
        k2, _, _ = orc.dequant_page(b2, 32, lo_bit=4)
        k4, vh, _ = orc.dequant_page(b4, 32, lo_bit=4, v_bit=4)
        assert (k2 == k4).all()
        assert (vh == _np_value_quant(xv, 15)[0]).all()


def test_value_closed_forms(orc):
    """Value groups on a power-of-two grid {0..15} * delta decode exactly, and a
    constant group decodes exactly with step 0."""
    r = _rng(3)
    xv = np.zeros((32, 128), np.float32)
    for t in range(32):
        for G in range(4):
            off = float(r.integers(-4, 4))
            g = slice(32 * G, 32 * G + 32)
            if (t + G) % 5 == 0:
                xv[t, g] = off + 0.5
            else:
                xv[t, g] = off + 0.125 * r.integers(0, 16, 32)
                xv[t, 32 * G], xv[t, 32 * G + 1] = off, off + 0.125 * 15
    xk, _ = _kv(11)
    blob, st = orc.quantize_page_f32(xk, xv, 0, lo_bit=4, v_bit=4)
    _, vh, _ = orc.dequant_page(blob, 0, lo_bit=4, v_bit=4)
    assert st == 0
    assert (vh == xv.astype(np.float64)).all()


def test_wider_values_never_lose(orc):
    """The 4-bit Value grid contains the 2-bit grid (j = 5k) over the same range:
    every Value element is reconstructed at least as well with 4-bit Values, up
    to the rounding of the stored steps, and the total error is far lower."""
    tot2 = tot4 = 0.0
    for seed in range(20, 26):
        xk, xv = _kv(seed)
        b2, _ = orc.quantize_page_f32(xk, xv, 0, lo_bit=4)
        b4, _ = orc.quantize_page_f32(xk, xv, 0, lo_bit=4, v_bit=4)
        _, v2, _ = orc.dequant_page(b2, 0, lo_bit=4)
        _, v4, _ = orc.dequant_page(b4, 0, lo_bit=4, v_bit=4)
        x = xv.astype(np.float64)
        e2, e4 = np.abs(v2 - x), np.abs(v4 - x)
        g = x.reshape(32, 4, 32)
        rng = np.repeat((g.max(2) - g.min(2))[:, :, None], 32, 2).reshape(32, 128)
        assert (e4 <= e2 + 2.0 ** -6 * rng + 1e-6).all()
        tot2 += float((e2 ** 2).sum())
        tot4 += float((e4 ** 2).sum())
    assert tot4 < tot2 / 15


def test_attention_v4_against_numpy(orc):
    """Decode attention with 4-bit Values equals fp64 softmax attention written
    here over the oracle's own dequantized pages (brute force, tiny case), for
    uniform 4-bit KV and for Kitty (8, 4) Keys."""
    for n_hi in (0, 32):
        B, Hkv, Hq = 2, 1, 2
        w = synth.Workload("pv4", B, Hq, Hkv, n_hi, synth.BF16, np.array([2, 3]), np.array([5, 0]))
        inp = synth.host_inputs(w, seed=4)
        per_page = orc.page_bytes(n_hi, 4, 4) * Hkv
        pool = np.zeros(inp["pool_pages"] * per_page, np.uint8)
        assert orc.quantize_pages(Hkv, n_hi, 0, synth.BF16, inp["k"], inp["v"], inp["page_ids"],
                                  pool, inp["pool_pages"], lo_bit=4, v_bit=4) == 0
        sm = float(np.float32(1 / math.sqrt(128)))
        out, st = orc.decode_attention(Hkv, Hq, n_hi, synth.BF16, inp["q"], pool,
                                       inp["pool_pages"], inp["block_table"], inp["num_pages"],
                                       inp["tail_k"], inp["tail_v"], inp["tail_len"], sm,
                                       lo_bit=4, v_bit=4)
        assert st == 0
        for b in range(B):
            ks, vs = [], []
            for p in range(int(inp["num_pages"][b])):
                pid = int(inp["block_table"][b, p])
                kh, vh, _ = orc.dequant_page(pool[pid * per_page:(pid + 1) * per_page], n_hi,
                                             lo_bit=4, v_bit=4)
                ks.append(kh)
                vs.append(vh)
            tl = int(inp["tail_len"][b])
            ks.append(synth.from_bits(inp["tail_k"][b, 0, :tl], synth.BF16).astype(np.float64))
            vs.append(synth.from_bits(inp["tail_v"][b, 0, :tl], synth.BF16).astype(np.float64))
            K, V = np.concatenate(ks), np.concatenate(vs)
            for h in range(Hq):
                q = synth.from_bits(inp["q"][b, h], synth.BF16).astype(np.float64)
                s = sm * (K @ q)
                p = np.exp(s - s.max())
                assert np.allclose(out[b, h], (p @ V) / p.sum(), rtol=1e-12, atol=1e-12)


def test_append_equals_bulk_with_4bit_values(orc):
    """Token-by-token append with flushes writes the same pages as bulk
    quantization of the same tokens (page mode), with 4-bit Values."""
    Hkv, n_hi, P = 2, 0, 32
    r = _rng(5)
    k = synth.to_bits(r.standard_normal((2 * P, Hkv, 128)) * np.exp(r.standard_normal(128)),
                      synth.BF16)
    v = synth.to_bits(r.standard_normal((2 * P, Hkv, 128)), synth.BF16)
    per_page = orc.page_bytes(n_hi, 4, 4) * Hkv
    bulk = np.zeros(2 * per_page, np.uint8)
    assert orc.quantize_pages(Hkv, n_hi, 0, synth.BF16, k, v, np.array([0, 1], np.int32), bulk, 2,
                              lo_bit=4, v_bit=4) == 0
    pool = np.zeros(2 * per_page, np.uint8)
    tail_k = np.zeros((1, Hkv, P, 128), np.uint16)
    tail_v = np.zeros_like(tail_k)
    tail_len = np.zeros(1, np.int32)
    bt = np.full((1, 2), -1, np.int32)
    npg = np.zeros(1, np.int32)
    rs = np.zeros((1, Hkv, 128), np.float32)
    rq = np.zeros_like(rs)
    rc = np.zeros((1, Hkv), np.int32)
    for t in range(2 * P):
        fl = np.array([t // P if t % P == P - 1 else -1], np.int32)
        assert orc.append_token(Hkv, n_hi, 0, synth.BF16, k[t][None], v[t][None], tail_k, tail_v,
                                tail_len, rs, rq, rc, fl, bt, 2, npg, pool, 2, lo_bit=4,
                                v_bit=4) == 0
    assert (bt == [[0, 1]]).all() and int(npg[0]) == 2 and int(tail_len[0]) == 0
    assert (pool == bulk).all()
