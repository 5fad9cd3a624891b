"""Pins of the oracle's (hi_bit, lo_bit) = (8, 4) configuration (VeloxQuant-MLX
docs, "Tuning avg_bits": the (0.25, 8, 4) row, 5.0 Key bits): Key channels at
4 bits, boosted channels at 8 bits split into two uniform 4-bit planes (the
paper abstract's two-uniform-tensor decomposition with 4-bit planes).

Each pin checks the oracle against an independent statement of the same fact:
a per-channel quantizer written here from its textbook definition, closed
forms, brute force over the plane maps, and the grid inclusion that orders the
errors of the two configurations.
"""

import numpy as np

from mixed_precision_bit_gb300 import synth
from tests.test_oracle_pins import np_step


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16(x):
    return synth.from_bits(synth.to_bits(np.asarray(x, np.float32), synth.BF16), synth.BF16)


def _kv(seed):
    r = _rng(seed)
    sig = np.exp(r.standard_normal(128))
    return _bf16(r.standard_normal((32, 128)) * sig), _bf16(r.standard_normal((32, 128)))


def _np_quant(x, levels, factor=1):
    """Per-channel asymmetric min/max quantizer over 32 tokens: fp16 minimum,
    step stored as np_step(factor * s) and used as that / factor, codes
    rint((x - M) * (1/u)) in fp32, clamp to [0, levels]."""
    x = x.astype(np.float32)
    mn, mx = x.min(0), x.max(0)
    M = mn.astype(np.float16).astype(np.float32)
    s = ((mx - mn).astype(np.float32) / np.float32(levels)).astype(np.float32)
    u = np_step(s * np.float32(factor)) / np.float32(factor)
    with np.errstate(divide="ignore", invalid="ignore"):
        ru = np.where(u == 0, np.float32(0), np.float32(1) / np.where(u == 0, np.float32(1), u))
        code = np.clip(np.rint((x - M).astype(np.float32) * ru.astype(np.float32)), 0, levels)
    code = np.where(u == 0, 0, code)
    return M.astype(np.float64) + u.astype(np.float64) * code, code.astype(np.int64)


def test_page_bytes_84(orc):
    """Kbase 2048 B (4 bits x 128 x 32), Kextra 16 B per boosted row, the rest as
    in the (4, 2) format: 4096 + 17 * n_hi."""
    for nh in (0, 16, 32, 64, 128):
        assert orc.page_bytes(nh, 4) == 2048 + 16 * nh + 512 + nh + 1024 + 512
    assert orc.page_bytes(32, 3) == -1


def test_nibble_maps_are_bijections(orc):
    seen = {orc.key_pos4(c, t, 16) for c in range(128) for t in range(32)}
    assert len(seen) == 4096 and {w for w, _ in seen} == set(range(512))
    assert {b for _, b in seen} == set(range(2, 32, 4))   # nibble starts, rotated by 2
    for nh in (16, 32, 128):
        seen = {orc.key_pos4(j, t, 2 * (nh // 16)) for j in range(nh) for t in range(32)}
        assert len(seen) == nh * 32 and max(w for w, _ in seen) == nh * 4 - 1


def test_hf0_is_uniform_4bit(orc):
    """n_hi = 0 at lo_bit 4 is uniform 4-bit per-channel Key quantization."""
    for seed in range(8):
        xk, xv = _kv(seed)
        blob, st = orc.quantize_page_f32(xk, xv, 0, lo_bit=4)
        kh, _, st2 = orc.dequant_page(blob, 0, lo_bit=4)
        want, _ = _np_quant(xk, 15)
        assert st == 0 and st2 == 0
        assert (kh == want).all()


def test_hf1_is_uniform_8bit(orc):
    """n_hi = 128 at lo_bit 4: every channel 8-bit, the stored base-plane step is
    16 x the 8-bit step (power-of-two scaling commutes with fp16 rounding for
    normal halves)."""
    for seed in range(8):
        xk, xv = _kv(seed + 20)
        blob, _ = orc.quantize_page_f32(xk, xv, 128, lo_bit=4)
        kh, _, _ = orc.dequant_page(blob, 128, lo_bit=4)
        want, _ = _np_quant(xk, 255, factor=16)
        assert (kh == want).all()


def _planes4(orc, blob, n_hi):
    def nib(off, w, b):
        x = int.from_bytes(bytes(blob[off + 4 * w:off + 4 * w + 4]), "little")
        return ((x >> b) | (x << (32 - b))) & 15   # a nibble at bit 30 wraps to bit 0
    base = np.array([[nib(0, *orc.key_pos4(c, t, 16)) for c in range(128)] for t in range(32)])
    extra = np.array([[nib(2048, *orc.key_pos4(j, t, 2 * (n_hi // 16))) for j in range(n_hi)]
                      for t in range(32)]).reshape(32, n_hi)
    return base, extra


def test_planes_recombine_to_8bit_code(orc):
    """16 * hi + lo is the boosted channel's 8-bit code; normal channels hold
    their 4-bit code in the base plane."""
    xk, xv = _kv(31)
    blob, _ = orc.quantize_page_f32(xk, xv, 32, lo_bit=4)
    base, extra = _planes4(orc, blob, 32)
    kch = orc.page_channels(blob, 32, lo_bit=4).astype(np.int64)
    assert (np.diff(kch) > 0).all()
    _, code8 = _np_quant(xk, 255, factor=16)
    for j, c in enumerate(kch):
        assert (16 * base[:, c] + extra[:, j] == code8[:, c]).all()
    normal = np.setdiff1d(np.arange(128), kch)
    _, code4 = _np_quant(xk, 15)
    assert (base[:, normal] == code4[:, normal]).all()


def test_closed_forms_84(orc):
    """Values on a power-of-two grid {0..255}*delta (boosted) and {0..15}*delta
    decode exactly; constant channels decode exactly."""
    r = _rng(7)
    xk = np.zeros((32, 128), np.float32)
    for c in range(128):
        off = float(r.integers(-8, 8))
        if c < 32:       # high variance: boosted, 256-level grid of step 2^-1
            xk[:, c] = off + 0.5 * r.integers(0, 256, 32)
            xk[0, c], xk[1, c] = off, off + 0.5 * 255
        elif c < 48:     # constant
            xk[:, c] = off + 0.25
        else:            # 16-level grid of step 2^-4
            xk[:, c] = off + 0.0625 * r.integers(0, 16, 32)
            xk[0, c], xk[1, c] = off, off + 0.0625 * 15
    xv = np.tile(np.array([0, 1, 2, 3] * 32, np.float32) * 0.5, (32, 1))
    blob, st = orc.quantize_page_f32(xk, xv, 32, lo_bit=4)
    kh, vh, _ = orc.dequant_page(blob, 32, lo_bit=4)
    assert st == 0
    assert set(orc.page_channels(blob, 32, lo_bit=4).tolist()) == set(range(32))
    assert (kh == xk.astype(np.float64)).all()
    assert (vh == xv.astype(np.float64)).all()


def test_wider_planes_never_lose(orc):
    """The 4-bit grid contains the 2-bit grid (j = 5k) and the 8-bit grid the 4-bit
    one (j = 17k), over the same range: with the same boost set every Key element
    is reconstructed at least as well at (8, 4) as at (4, 2), up to the fp16
    rounding of the stored steps; the total error is far lower.  Values are the
    same 2-bit format in both."""
    tot42 = tot84 = 0.0
    for seed in range(40, 48):
        xk, xv = _kv(seed)
        b42, _ = orc.quantize_page_f32(xk, xv, 32)
        b84, _ = orc.quantize_page_f32(xk, xv, 32, lo_bit=4)
        assert (orc.page_channels(b42, 32) == orc.page_channels(b84, 32, lo_bit=4)).all()
        k42, v42, _ = orc.dequant_page(b42, 32)
        k84, v84, _ = orc.dequant_page(b84, 32, lo_bit=4)
        x = xk.astype(np.float64)
        e42, e84 = np.abs(k42 - x), np.abs(k84 - x)
        # rounding of the stored steps: each is at most 2^-6 above its exact
        # step, which moves the coarser grid's top point by at most 2^-6 * range
        slack = 2.0 ** -6 * (x.max(0) - x.min(0)) + 1e-6
        assert (e84 <= e42 + slack).all()
        assert (v42 == v84).all()
        tot42 += float((e42 ** 2).sum())
        tot84 += float((e84 ** 2).sum())
    assert tot84 < tot42 / 20


def test_attention_84_against_numpy(orc):
    """Decode attention in the (8, 4) format equals fp64 softmax attention written
    here over the oracle's own dequantized pages (brute force, tiny case)."""
    import math
    B, Hkv, Hq, n_hi = 2, 1, 2, 32
    w = synth.Workload("p84", B, Hq, Hkv, n_hi, synth.BF16, np.array([2, 3]), np.array([5, 0]))
    inp = synth.host_inputs(w, seed=3)
    per_page = orc.page_bytes(n_hi, 4) * Hkv
    pool = np.zeros(inp["pool_pages"] * per_page, np.uint8)
    assert orc.quantize_pages(Hkv, n_hi, 0, synth.BF16, inp["k"], inp["v"], inp["page_ids"], pool,
                              inp["pool_pages"], lo_bit=4) == 0
    sm = float(np.float32(1 / math.sqrt(128)))   # the API takes sm_scale in fp32
    out, st = orc.decode_attention(Hkv, Hq, n_hi, synth.BF16, inp["q"], pool, inp["pool_pages"],
                                   inp["block_table"], inp["num_pages"], inp["tail_k"],
                                   inp["tail_v"], inp["tail_len"], sm, lo_bit=4)
    assert st == 0
    for b in range(B):
        ks, vs = [], []
        for p in range(int(inp["num_pages"][b])):
            pid = int(inp["block_table"][b, p])
            kh, vh, _ = orc.dequant_page(pool[pid * per_page:(pid + 1) * per_page], n_hi, lo_bit=4)
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
