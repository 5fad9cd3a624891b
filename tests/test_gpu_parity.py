"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Packed pages, channel lists, scales and running
statistics must be bit-exact; attention within 2e-3 * RMS(oracle output)
(+ half an output ulp for 16-bit outputs)."""

import dataclasses

import numpy as np
import pytest

import oracle
from mixed_precision_bit_gb300 import synth
from tests.kitty_cases import (attn_error, gpu_decode, gpu_quantize, oracle_decode,
                               oracle_quantize, dev16, dev32, cfg_for)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixed_precision_bit_gb300 import kitty
    kitty.load()


def _variant(name, **kw):
    return dataclasses.replace(synth.workload(name), **kw)


CASES = [
    ("tiny", {}),
    ("small_gqa", {}),
    ("small_gqa", dict(n_hi=0)),
    ("small_gqa", dict(n_hi=16)),
    ("small_gqa", dict(n_hi=64)),
    ("small_gqa", dict(n_hi=128)),
    ("small_gqa", dict(dtype=synth.F16)),
    ("small_gqa", dict(Hq=2, Hkv=2)),            # g = 1
    ("small_gqa", dict(Hq=6, Hkv=3)),            # g = 2
    ("small_gqa", dict(Hq=6, Hkv=2)),            # g = 3
    ("small_gqa", dict(Hq=16, Hkv=2)),           # g = 8: two head-group CTAs
    ("small_gqa", dict(Hq=10, Hkv=2, n_hi=16)),  # g = 5: a group of 4 and one of 1
    ("small_gqa", dict(Hq=12, Hkv=1, dtype=synth.F16)),  # g = 12
    # (hi_bit, lo_bit) = (8, 4): two 4-bit Key planes
    ("tiny", dict(lo_bit=4)),
    ("small_gqa", dict(lo_bit=4)),
    ("small_gqa", dict(lo_bit=4, n_hi=0)),
    ("small_gqa", dict(lo_bit=4, n_hi=48)),
    ("small_gqa", dict(lo_bit=4, n_hi=128)),
    ("small_gqa", dict(lo_bit=4, dtype=synth.F16, n_hi=16, Hq=6, Hkv=3)),
    # 4-bit Values: uniform 4-bit KV (n_hi = 0) and Kitty (8, 4) Keys
    ("tiny", dict(lo_bit=4, v_bit=4)),
    ("small_gqa", dict(lo_bit=4, v_bit=4, n_hi=0)),
    ("small_gqa", dict(lo_bit=4, v_bit=4)),
    ("small_gqa", dict(lo_bit=4, v_bit=4, n_hi=128, dtype=synth.F16)),
    ("small_gqa", dict(lo_bit=4, v_bit=4, n_hi=16, Hq=6, Hkv=2)),
    ("small_gqa", dict(lo_bit=4, v_bit=4, n_hi=0, Hq=16, Hkv=2)),
]


def _ids(c):
    return c[0] + "".join("-%s%s" % kv for kv in c[1].items())


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_quantize_bit_exact(case):
    w = _variant(case[0], **case[1])
    inp = synth.host_inputs(w, seed=1)
    pool, _ = gpu_quantize(w, inp)
    ref, _, st = oracle_quantize(w, inp)
    assert st == 0
    got = pool.cpu().numpy()
    assert got.shape == ref.shape
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, "first mismatching bytes at %s" % bad[:8]


def _signed_zeros(inp):
    """Plant +0 / -0 (16-bit 0x0000 / 0x8000) into Key channels and Value groups
    of page 0, head 0, where they decide a minimum or a maximum."""
    P, Z, N = 0x0000, 0x8000, None
    k, v = inp["k"], inp["v"]
    t = np.arange(32)
    k[t, 0, 3] = np.where(t % 2 == 0, P, Z)          # all zeros, +0 first
    k[t, 0, 4] = np.where(t % 2 == 0, Z, P)          # all zeros, -0 first
    k[t, 0, 5] = np.where(t < 16, np.where(t % 2 == 0, P, Z), k[t, 0, 5] & 0x7FFF)  # min is a zero
    k[t, 0, 6] = np.where(t < 16, np.where(t % 2 == 0, Z, P), k[t, 0, 6] | 0x8000)  # max is a zero
    c = np.arange(32)
    v[0, 0, c] = np.where(c % 2 == 0, P, Z)          # token 0, group 0: zeros, +0 first
    v[1, 0, 32 + c] = np.where(c % 2 == 0, Z, P)     # token 1, group 1: zeros, -0 first
    v[2, 0, 64 + c] = np.where(c < 8, np.where(c % 2 == 0, Z, P), v[2, 0, 64 + c] & 0x7FFF)
    v[3, 0, 96 + c] = np.where(c < 8, np.where(c % 2 == 0, P, Z), v[3, 0, 96 + c] | 0x8000)
    return inp


@pytest.mark.parametrize("lo_bit,v_bit", [(2, 2), (4, 2), (4, 4)], ids=["42", "84", "84v4"])
@pytest.mark.parametrize("mode", [0, 1], ids=["page", "running"])
@pytest.mark.parametrize("dtype", [synth.BF16, synth.F16], ids=["bf16", "f16"])
def test_quantize_signed_zeros_bit_exact(dtype, mode, lo_bit, v_bit):
    """A minimum or maximum that is a signed zero is stored with the sign the
    IEEE 754-2019 minimum and maximum give, whatever the token order: of +0 and
    -0 the minimum is -0 and the maximum +0 (Value groups: also with 4-bit
    Values, whose min and max run on packed 16-bit pairs)."""
    w = _variant("small_gqa", dtype=dtype, lo_bit=lo_bit, v_bit=v_bit)
    inp = _signed_zeros(synth.host_inputs(w, seed=1))
    pool, run = gpu_quantize(w, inp, mode=mode)
    ref, ref_run, st = oracle_quantize(w, inp, mode=mode)
    assert st == 0
    got = pool.cpu().numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, "first mismatching bytes at %s" % bad[:8]


@pytest.mark.parametrize("lo_bit,v_bit", [(2, 2), (4, 2), (4, 4)], ids=["42", "84", "84v4"])
@pytest.mark.parametrize("mode", [1, 2], ids=["running", "sequence"])
def test_quantize_running_bit_exact(mode, lo_bit, v_bit):
    w = _variant("small_gqa", pages=np.array([5, 3, 9]), drift=64, lo_bit=lo_bit, v_bit=v_bit)
    inp = synth.host_inputs(w, seed=2)
    pool, run = gpu_quantize(w, inp, mode=mode)
    ref, (rs, rq, rc), st = oracle_quantize(w, inp, mode=mode)
    assert st == 0
    assert (pool.cpu().numpy() == ref).all()
    assert (run[0].cpu().numpy().view(np.uint32) == rs.view(np.uint32)).all()
    assert (run[1].cpu().numpy().view(np.uint32) == rq.view(np.uint32)).all()
    assert (run[2].cpu().numpy() == rc).all()


@pytest.mark.parametrize("mode", [1, 2], ids=["running", "sequence"])
def test_quantize_running_many_chains_bit_exact(mode):
    """Enough (sequence, kv head) chains for the fused statistics walk (at least
    3 per SM): pages, channel lists and accumulators bit-exact with the oracle,
    as on the three-launch path the small cases take."""
    import torch
    chains = 3 * torch.cuda.get_device_properties(0).multi_processor_count
    B = (chains + 1) // 2 + 8
    pages = (synth.bits(9, "walk/pages", B) % np.uint64(4)).astype(np.int64) + 1
    pages[5] = 0                                    # a sequence without pages
    w = _variant("small_gqa", B=B, pages=pages, tails=np.zeros(B, np.int64), drift=64)
    assert w.B * w.Hkv >= chains
    inp = synth.host_inputs(w, seed=3)
    pool, run = gpu_quantize(w, inp, mode=mode)
    ref, (rs, rq, rc), st = oracle_quantize(w, inp, mode=mode)
    assert st == 0
    assert (pool.cpu().numpy() == ref).all()
    assert (run[0].cpu().numpy().view(np.uint32) == rs.view(np.uint32)).all()
    assert (run[1].cpu().numpy().view(np.uint32) == rq.view(np.uint32)).all()
    assert (run[2].cpu().numpy() == rc).all()


def test_decode_with_plan_hint():
    """The total-pages planning hint changes only the split layout: a ragged
    batch decodes within tolerance with the exact, a stale and a large hint."""
    import torch
    from mixed_precision_bit_gb300 import kitty
    w = _variant("small_gqa", pages=np.array([37, 1, 90]), tails=np.array([0, 5, 17]))
    inp = synth.host_inputs(w, seed=8)
    pool, _ = gpu_quantize(w, inp)
    ref, _ = oracle_decode(w, inp, pool.cpu().numpy())
    hints = [(int(w.pages.sum()), 0), (5, 0), (100000, 0),
             (int(w.pages.sum()), int(w.pages.max())), (int(w.pages.sum()), 3), (0, 100000)]
    for hint, mx in hints:
        cfg = cfg_for(w)
        cfg.decode_total_pages = hint
        cfg.decode_max_pages = mx
        bt = inp["block_table"]
        ws = torch.empty(max(kitty.decode_workspace_bytes(cfg, w.B, bt.shape[1]), 16) // 4,
                         dtype=torch.float32, device="cuda")
        out = torch.empty((w.B, w.Hq, 128), dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        kitty.decode_attention(cfg, dev16(inp["q"]), pool, inp["pool_pages"], dev32(bt),
                               dev32(inp["num_pages"]), dev16(inp["tail_k"]), dev16(inp["tail_v"]),
                               dev32(inp["tail_len"]), float(np.float32(1 / np.sqrt(128))), out,
                               workspace=ws, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        excess, rel = attn_error(out.cpu().numpy().astype(np.float64), ref)
        assert excess <= 0, "hint %d: max err %.3e of RMS" % (hint, rel)


def test_quantize_bad_seq_status():
    """A seq_of_page entry outside [0, n_seqs) is reported; the other pages of
    the batch are quantized as usual (bit-exact with a batch without the bad
    page)."""
    import torch
    from mixed_precision_bit_gb300 import kitty
    w = _variant("small_gqa", pages=np.array([4, 2, 3]))
    inp = synth.host_inputs(w, seed=6)
    good, _ = gpu_quantize(w, inp, mode=1)
    bad_seq = inp["seq_of_page"].copy()
    bad_seq[-1] = w.B          # the last page claims a sequence that does not exist
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    inp2 = dict(inp, seq_of_page=bad_seq)
    pool, _ = gpu_quantize(w, inp2, mode=1, status=st)
    assert int(st.item()) == kitty.ST["BAD_SEQ"]
    per_page = kitty.page_bytes(cfg_for(w, rank_mode=1))[1]
    ids = inp["page_ids"]
    g, p = good.cpu().numpy(), pool.cpu().numpy()
    for i in range(ids.size - 1):
        sl = slice(int(ids[i]) * per_page, (int(ids[i]) + 1) * per_page)
        assert (g[sl] == p[sl]).all(), i
    sl = slice(int(ids[-1]) * per_page, (int(ids[-1]) + 1) * per_page)
    assert not p[sl].any()     # never written (the pool starts zeroed)


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16", "f16"])
def test_decode_attention(case, out_dtype):
    w = _variant(case[0], **case[1])
    inp = synth.host_inputs(w, seed=3)
    pool, _ = gpu_quantize(w, inp)
    got = gpu_decode(w, inp, pool, out_dtype)
    ref, st = oracle_decode(w, inp, pool.cpu().numpy())
    excess, rel = attn_error(got, ref, out_dtype)
    assert excess <= 0, "max err %.3e of RMS" % rel


@pytest.mark.parametrize("out_dtype", ["f32", "bf16", "f16"])
def test_decode_unaligned_output(out_dtype):
    """An output array that starts one element past a 16-byte boundary (a plain
    contiguous view) gets the same values as an aligned one: the split merge
    stores vectors only into aligned arrays, and the one-split path stores
    scalars."""
    w = _variant("small_gqa", pages=np.array([37, 1, 64]), tails=np.array([0, 5, 17]))
    inp = synth.host_inputs(w, seed=4)
    pool, _ = gpu_quantize(w, inp)
    for pps in (4, 0, 64):  # a 16-split merge, the planner's splits, one split
        a = gpu_decode(w, inp, pool, out_dtype, pps=pps)
        b = gpu_decode(w, inp, pool, out_dtype, pps=pps, out_offset=1)
        assert not np.isnan(a).any() and np.array_equal(a, b), pps


@pytest.mark.parametrize("Hq", [8, 16], ids=["g4", "g8"])
@pytest.mark.parametrize("pps", [1, 3, 4, 5, 64])
def test_decode_split_invariance(pps, Hq):
    """Different split-K chunks agree to well inside the tolerance.  They are not
    identical: probabilities enter the tensor cores as fp16 hi/lo pairs relative to
    each warp's running max, so tiny weights fall in the fp16 subnormal range with
    a different absolute rounding per split layout (~1e-5 of RMS observed).  On
    the 64-page sequence the chunk sizes give 64, 22, 16, 13 and 1 splits: the
    merge's several-round path (full and ragged last round), its one-round path
    and no merge at all; the shorter sequences leave splits without pages.  With
    g = 8 the same holds for the kernel that carries 8 query heads per CTA."""
    w = _variant("small_gqa", Hq=Hq, pages=np.array([37, 1, 64]), tails=np.array([0, 5, 17]))
    inp = synth.host_inputs(w, seed=4)
    pool, _ = gpu_quantize(w, inp)
    a = gpu_decode(w, inp, pool, pps=pps)
    c = gpu_decode(w, inp, pool, pps=0)
    scale = np.sqrt(np.mean(c ** 2))
    assert np.abs(a - c).max() <= 1e-4 * scale
    ref, _ = oracle_decode(w, inp, pool.cpu().numpy())
    assert attn_error(a, ref)[0] <= 0


@pytest.mark.parametrize("Hq", [8, 16, 12], ids=["g4", "g8", "g6"])
def test_decode_ragged_and_empty(Hq):
    """Sequences with only a tail, only pages, nothing at all, and a full tail."""
    w = _variant("small_gqa", Hq=Hq, B=5, pages=np.array([0, 3, 0, 6, 1]),
                 tails=np.array([9, 0, 0, 32 - 1, 0]))
    inp = synth.host_inputs(w, seed=5)
    inp["tail_len"][3] = 31
    pool, _ = gpu_quantize(w, inp)
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = gpu_decode(w, inp, pool, status=st)
    ref, ost = oracle_decode(w, inp, pool.cpu().numpy())
    assert ost == oracle.ST["EMPTY"] and int(st.item()) == oracle.ST["EMPTY"]
    assert (got[2] == 0).all()
    assert attn_error(got, ref)[0] <= 0


@pytest.mark.parametrize("Hq", [1, 8], ids=["g1", "g8"])
def test_decode_bad_page_sets_status(Hq):
    w = _variant("tiny", Hq=Hq)
    inp = synth.host_inputs(w, seed=6)
    pool, _ = gpu_quantize(w, inp)
    inp["block_table"][0, 3] = 10 ** 6
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_decode(w, inp, pool, status=st)
    assert int(st.item()) == oracle.ST["BAD_PAGE"]


def test_quantize_range_status():
    w = synth.workload("tiny")
    inp = synth.host_inputs(w, seed=7)
    inp["k"][5, 0, 9] = np.float32(70000.0).astype(np.float16).view(np.uint16)  # fp16 inf
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_quantize(w, inp, status=st)
    assert int(st.item()) == oracle.ST["NONFINITE"]


def test_append_matches_oracle():
    """Token-by-token append with running statistics and flushes, bit-exact
    pages/state, then decode over the resulting cache."""
    import torch
    from mixed_precision_bit_gb300 import kitty
    B, Hkv, Hq, n_hi, steps = 3, 2, 8, 32, 70
    w = synth.Workload("append", B, Hq, Hkv, n_hi, synth.BF16, np.zeros(B, np.int64),
                       np.array([30, 0, 12]))
    cfg = cfg_for(w, rank_mode=1)
    r = np.random.default_rng(9)
    max_pages = 4
    pool_pages = B * max_pages
    blob, per_page = kitty.page_bytes(cfg)
    # oracle state
    o = dict(tail_k=np.zeros((B, Hkv, 32, 128), np.uint16), tail_len=np.array([30, 0, 12], np.int32),
             run_sum=np.zeros((B, Hkv, 128), np.float32), run_count=np.zeros((B, Hkv), np.int32),
             block_table=np.full((B, max_pages), -1, np.int32), num_pages=np.zeros(B, np.int32),
             pool=np.zeros(pool_pages * per_page, np.uint8))
    o["tail_v"] = o["tail_k"].copy()
    o["run_sumsq"] = o["run_sum"].copy()
    pre = synth.to_bits(r.standard_normal((B, Hkv, 32, 128)), synth.BF16)
    o["tail_k"][:] = pre
    o["tail_v"][:] = pre[::-1]
    g = {k: (torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).cuda())
         for k, v in o.items()}
    alloc = kitty.PageAllocator(pool_pages)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sig = np.exp(r.standard_normal(128))
    for step in range(steps):
        kn = synth.to_bits(r.standard_normal((B, Hkv, 128)) * sig, synth.BF16)
        vn = synth.to_bits(r.standard_normal((B, Hkv, 128)), synth.BF16)
        fl = np.full(B, -1, np.int32)
        for b in range(B):
            if o["tail_len"][b] + 1 == 32 and o["num_pages"][b] < max_pages:
                fl[b] = alloc.alloc(1)[0]
        s1 = oracle.append_token(Hkv, n_hi, 1, synth.BF16, kn, vn, o["tail_k"], o["tail_v"],
                                 o["tail_len"], o["run_sum"], o["run_sumsq"], o["run_count"], fl,
                                 o["block_table"], max_pages, o["num_pages"], o["pool"], pool_pages)
        assert s1 == 0
        kitty.append_token(cfg, dev16(kn), dev16(vn), g["tail_k"], g["tail_v"], g["tail_len"],
                           g["run_sum"], g["run_sumsq"], g["run_count"], dev32(fl),
                           g["block_table"], g["num_pages"], g["pool"], pool_pages, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for k, v in o.items():
        gv = g[k].cpu().numpy()
        if v.dtype == np.uint16:
            gv = gv.view(np.uint16)
        assert (gv.view(np.uint8) == v.view(np.uint8)).all(), k
    assert (o["num_pages"] > 0).all()
    inp = dict(q=synth.to_bits(r.standard_normal((B, Hq, 128)), synth.BF16), pool_pages=pool_pages,
               block_table=o["block_table"], num_pages=o["num_pages"], tail_k=o["tail_k"],
               tail_v=o["tail_v"], tail_len=o["tail_len"])
    got = gpu_decode(w, inp, g["pool"])
    ref, _ = oracle_decode(w, inp, o["pool"])
    assert attn_error(got, ref)[0] <= 0


def test_determinism():
    """Two runs of the same quantize and decode give bitwise-equal pools and outputs
    (fixed split layout, fixed combine order, no atomics on data)."""
    for mode in (0, 1):
        w = _variant("small_gqa", pages=np.array([33, 2, 40]), tails=np.array([9, 0, 31]))
        inp = synth.host_inputs(w, seed=12)
        pa, _ = gpu_quantize(w, inp, mode=mode)
        pb, _ = gpu_quantize(w, inp, mode=mode)
        assert (pa.cpu().numpy() == pb.cpu().numpy()).all()
        oa = gpu_decode(w, inp, pa, pps=8)
        ob = gpu_decode(w, inp, pa, pps=8)
        assert (oa.view(np.uint64) == ob.view(np.uint64)).all()


@pytest.mark.parametrize("Hq", [8, 16, 10], ids=["g4", "g8", "g5"])
def test_grouped_heads_equal_single_head_calls(Hq):
    """A kv head's g query heads decoded together agree with g separate one-head
    calls over the same kv cache: query head hq reads kv head hq / g.  The split
    size is fixed, so both sides take the same splits."""
    w = _variant("small_gqa", Hq=Hq, Hkv=2, pages=np.array([12, 5, 20]), tails=np.array([3, 30, 0]))
    inp = synth.host_inputs(w, seed=13)
    pool, _ = gpu_quantize(w, inp)
    together = gpu_decode(w, inp, pool, pps=4)
    g = w.g
    for h in range(g):
        w1 = dataclasses.replace(w, Hq=w.Hkv)          # one query head per kv head
        inp1 = dict(inp, q=np.ascontiguousarray(inp["q"][:, h::g]))
        alone = gpu_decode(w1, inp1, pool, pps=4)
        ref = together[:, h::g]
        scale = np.sqrt(np.mean(ref ** 2))
        assert np.abs(alone - ref).max() <= 1e-6 * scale, h
