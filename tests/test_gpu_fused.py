"""GPU parity of the fused decode step (kitty_append_decode): against the
oracle's append_token followed by decode_attention on the same seeded inputs,
step by step, with flushes (pages, tails, running statistics, block table and
lengths bit-exact; attention within 2e-3 * RMS), and against the library's two
separate calls."""

import math

import numpy as np
import pytest

import oracle
from mixed_precision_bit_gb300 import synth
from tests.kitty_cases import attn_error, cfg_for, dev16, dev32

pytestmark = pytest.mark.gpu

SM = float(np.float32(1 / math.sqrt(128)))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixed_precision_bit_gb300 import kitty
    kitty.load()


def _initial(mode, dtype, pages, tails, Hkv=2, Hq=8, n_hi=32, extra=3, seed=11, lo_bit=2, v_bit=2):
    """Oracle-built cache (prefilled pages quantized by the oracle, tails) with
    `extra` free block-table slots per sequence, as host arrays."""
    B = len(pages)
    w = synth.Workload("fused", B, Hq, Hkv, n_hi, dtype, np.asarray(pages), np.asarray(tails),
                       lo_bit=lo_bit, v_bit=v_bit)
    inp = synth.host_inputs(w, seed=seed)
    max_pages = int(max(pages)) + extra
    tot = int(np.sum(pages))
    pool_pages = tot + B * extra
    per_page = oracle.page_bytes(n_hi, lo_bit, v_bit) * Hkv
    st = dict(pool=np.zeros(pool_pages * per_page, np.uint8),
              block_table=np.full((B, max_pages), -1, np.int32),
              num_pages=np.asarray(pages, np.int32).copy(),
              tail_k=inp["tail_k"].copy(), tail_v=inp["tail_v"].copy(),
              tail_len=np.asarray(tails, np.int32).copy(),
              run_sum=np.zeros((B, Hkv, 128), np.float32), run_sumsq=np.zeros((B, Hkv, 128), np.float32),
              run_count=np.zeros((B, Hkv), np.int32))
    st["block_table"][:, :inp["block_table"].shape[1]] = inp["block_table"]
    if tot:
        kw = {}
        if mode != 0:
            kw = dict(seq_of_page=inp["seq_of_page"], n_seqs=B, run_sum=st["run_sum"],
                      run_sumsq=st["run_sumsq"], run_count=st["run_count"])
        assert oracle.quantize_pages(Hkv, n_hi, mode, dtype, inp["k"], inp["v"], inp["page_ids"],
                                     st["pool"], pool_pages, lo_bit=lo_bit, v_bit=v_bit, **kw) == 0
    return w, st, max_pages, pool_pages, tot


def _to_gpu(st):
    import torch
    return {k: torch.from_numpy((v.view(np.int16) if v.dtype == np.uint16 else v).copy()).cuda()
            for k, v in st.items()}


def _plan(st, max_pages, next_id):
    fl = np.full(st["tail_len"].size, -1, np.int32)
    for b in range(fl.size):
        if st["tail_len"][b] + 1 == 32 and st["num_pages"][b] < max_pages:
            fl[b] = next_id
            next_id += 1
    return fl, next_id


def _compare_state(o, g, keys=("pool", "tail_k", "tail_v", "tail_len", "num_pages", "block_table",
                               "run_sum", "run_sumsq", "run_count")):
    for k in keys:
        gv = g[k].cpu().numpy()
        assert (gv.view(np.uint8) == o[k].view(np.uint8)).all(), k


@pytest.mark.parametrize("mode,dtype,pps,lo_bit,v_bit",
                         [(1, synth.BF16, 0, 2, 2), (0, synth.BF16, 4, 2, 2),
                          (1, synth.F16, 1000, 2, 2), (2, synth.BF16, 2, 2, 2),
                          (1, synth.BF16, 4, 4, 2), (0, synth.F16, 1000, 4, 2),
                          (0, synth.BF16, 4, 4, 4), (1, synth.F16, 0, 4, 4)],
                         ids=["running-bf16", "page-bf16-splits", "running-f16-one-split",
                              "sequence-bf16-splits", "running-bf16-84", "page-f16-one-split-84",
                              "page-bf16-splits-kv4", "running-f16-84-v4"])
def test_fused_matches_oracle(mode, dtype, pps, lo_bit, v_bit):
    import torch
    from mixed_precision_bit_gb300 import kitty
    w, o, max_pages, pool_pages, next_id = _initial(mode, dtype, [5, 0, 9], [29, 31, 3],
                                                    lo_bit=lo_bit, v_bit=v_bit,
                                                    n_hi=0 if (mode, v_bit) == (0, 4) else 32)
    B, Hkv, Hq = w.B, w.Hkv, w.Hq
    cfg = cfg_for(w, rank_mode=mode, pps=pps)
    g = _to_gpu(o)
    ws = torch.empty(max(kitty.decode_workspace_bytes(cfg, B, max_pages), 16) // 4,
                     dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    r = np.random.default_rng(3 + mode)
    sig = np.exp(r.standard_normal(128))
    flushed = 0
    for step in range(36):
        kn = synth.to_bits(r.standard_normal((B, Hkv, 128)) * sig, dtype)
        vn = synth.to_bits(r.standard_normal((B, Hkv, 128)), dtype)
        q = synth.to_bits(r.standard_normal((B, Hq, 128)), dtype)
        fl, next_id = _plan(o, max_pages, next_id)
        flushed += int((fl >= 0).sum())
        assert oracle.append_token(Hkv, w.n_hi, mode, dtype, kn, vn, o["tail_k"], o["tail_v"],
                                   o["tail_len"], o["run_sum"], o["run_sumsq"], o["run_count"], fl,
                                   o["block_table"], max_pages, o["num_pages"], o["pool"],
                                   pool_pages, lo_bit=lo_bit, v_bit=v_bit) == 0
        ref, st = oracle.decode_attention(Hkv, Hq, w.n_hi, dtype, q, o["pool"], pool_pages,
                                          o["block_table"], o["num_pages"], o["tail_k"],
                                          o["tail_v"], o["tail_len"], SM, lo_bit=lo_bit,
                                          v_bit=v_bit)
        assert st == 0
        kitty.append_decode(cfg, dev16(kn), dev16(vn), dev16(q), g["tail_k"], g["tail_v"],
                            g["tail_len"], g["run_sum"], g["run_sumsq"], g["run_count"], dev32(fl),
                            g["block_table"], g["num_pages"], g["pool"], pool_pages, SM, out,
                            workspace=ws, status=status)
        got = out.cpu().numpy().astype(np.float64)
        excess, rel = attn_error(got, ref)
        assert excess <= 0, "step %d: max err %.3e of RMS" % (step, rel)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert flushed >= 3
    _compare_state(o, g)


def test_fused_equals_separate_calls():
    """Same cache, same inputs: the fused call and append_token + decode_attention
    leave bit-identical caches; outputs agree far inside the tolerance (the new
    page of a flush is summed in another order)."""
    import torch
    from mixed_precision_bit_gb300 import kitty
    w, o, max_pages, pool_pages, next_id = _initial(1, synth.BF16, [40, 3, 17], [31, 30, 0])
    B, Hkv, Hq = w.B, w.Hkv, w.Hq
    cfg = cfg_for(w, rank_mode=1, pps=8)
    ga, gb = _to_gpu(o), _to_gpu(o)
    ws = torch.empty(max(kitty.decode_workspace_bytes(cfg, B, max_pages), 16) // 4,
                     dtype=torch.float32, device="cuda")
    sa = torch.zeros(1, dtype=torch.int32, device="cuda")
    sb = torch.zeros(1, dtype=torch.int32, device="cuda")
    oa = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    ob = torch.empty_like(oa)
    r = np.random.default_rng(21)
    h_tail = o["tail_len"].copy()
    h_np = o["num_pages"].copy()
    for step in range(34):
        kn = dev16(synth.to_bits(r.standard_normal((B, Hkv, 128)), synth.BF16))
        vn = dev16(synth.to_bits(r.standard_normal((B, Hkv, 128)), synth.BF16))
        q = dev16(synth.to_bits(r.standard_normal((B, Hq, 128)), synth.BF16))
        fl, next_id = _plan(dict(tail_len=h_tail, num_pages=h_np), max_pages, next_id)
        full = fl >= 0
        h_tail = np.where(full, 0, h_tail + 1)
        h_np = h_np + full
        fld = dev32(fl)
        kitty.append_decode(cfg, kn, vn, q, ga["tail_k"], ga["tail_v"], ga["tail_len"],
                            ga["run_sum"], ga["run_sumsq"], ga["run_count"], fld,
                            ga["block_table"], ga["num_pages"], ga["pool"], pool_pages, SM, oa,
                            workspace=ws, status=sa)
        kitty.append_token(cfg, kn, vn, gb["tail_k"], gb["tail_v"], gb["tail_len"], gb["run_sum"],
                           gb["run_sumsq"], gb["run_count"], fld, gb["block_table"],
                           gb["num_pages"], gb["pool"], pool_pages, status=sb)
        kitty.decode_attention(cfg, q, gb["pool"], pool_pages, gb["block_table"], gb["num_pages"],
                               gb["tail_k"], gb["tail_v"], gb["tail_len"], SM, ob, workspace=ws,
                               status=sb)
        a, b = oa.cpu().numpy(), ob.cpu().numpy()
        assert np.abs(a - b).max() <= 1e-4 * np.sqrt(np.mean(b.astype(np.float64) ** 2)), step
    torch.cuda.synchronize()
    assert int(sa.item()) == 0 and int(sb.item()) == 0
    for k in ga:
        assert (ga[k].cpu().numpy().view(np.uint8) == gb[k].cpu().numpy().view(np.uint8)).all(), k


@pytest.mark.parametrize("case", ["tail_full", "bad_flush"])
def test_fused_status_codes(case):
    """Data errors give the separate calls' status and leave the same state."""
    import torch
    from mixed_precision_bit_gb300 import kitty
    ST = kitty.ST
    tails = [32, 4] if case == "tail_full" else [10, 4]
    w, o, max_pages, pool_pages, _ = _initial(0, synth.BF16, [6, 2], tails, extra=2)
    B, Hkv, Hq = w.B, w.Hkv, w.Hq
    cfg = cfg_for(w, rank_mode=0, pps=4)
    ga, gb = _to_gpu(o), _to_gpu(o)
    ws = torch.empty(max(kitty.decode_workspace_bytes(cfg, B, max_pages), 16) // 4,
                     dtype=torch.float32, device="cuda")
    r = np.random.default_rng(5)
    kn = dev16(synth.to_bits(r.standard_normal((B, Hkv, 128)), synth.BF16))
    vn = dev16(synth.to_bits(r.standard_normal((B, Hkv, 128)), synth.BF16))
    q = dev16(synth.to_bits(r.standard_normal((B, Hq, 128)), synth.BF16))
    fl = dev32(np.array([-1, -1] if case == "tail_full" else [8, -1], np.int32))
    sa = torch.zeros(1, dtype=torch.int32, device="cuda")
    sb = torch.zeros(1, dtype=torch.int32, device="cuda")
    oa = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    ob = torch.empty_like(oa)
    kitty.append_decode(cfg, kn, vn, q, ga["tail_k"], ga["tail_v"], ga["tail_len"], ga["run_sum"],
                        ga["run_sumsq"], ga["run_count"], fl, ga["block_table"], ga["num_pages"],
                        ga["pool"], pool_pages, SM, oa, workspace=ws, status=sa)
    kitty.append_token(cfg, kn, vn, gb["tail_k"], gb["tail_v"], gb["tail_len"], gb["run_sum"],
                       gb["run_sumsq"], gb["run_count"], fl, gb["block_table"], gb["num_pages"],
                       gb["pool"], pool_pages, status=sb)
    kitty.decode_attention(cfg, q, gb["pool"], pool_pages, gb["block_table"], gb["num_pages"],
                           gb["tail_k"], gb["tail_v"], gb["tail_len"], SM, ob, workspace=ws,
                           status=sb)
    torch.cuda.synchronize()
    want = ST["TAIL_FULL"] if case == "tail_full" else ST["BAD_FLUSH"]
    assert int(sa.item()) == want and int(sb.item()) == want
    for k in ga:
        assert (ga[k].cpu().numpy().view(np.uint8) == gb[k].cpu().numpy().view(np.uint8)).all(), k
    a, b = oa.cpu().numpy(), ob.cpu().numpy()
    assert np.abs(a - b).max() <= 1e-4 * np.sqrt(np.mean(b.astype(np.float64) ** 2))
