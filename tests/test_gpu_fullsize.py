"""Parity at the benchmark's full sizes and launch configuration, on sampled
sequences.  The workloads are built exactly as bench.py builds them (seeded K/V
generated on the GPU); the raw inputs of a few sequences are copied back and
given to the oracle, which quantizes them itself.  Checked: packed pages
bit-exact at their block-table page ids, decode attention of every head of the
sampled sequences within 2e-3 * RMS, and for the serving workload a few append
steps with flushes (running statistics) bit-exact."""

import math

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

SM = float(np.float32(1 / math.sqrt(128)))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _oracle_seq_pool(spec, k, v, running):
    """The oracle's pages for one sequence (local ids 0..np-1)."""
    n_hi, Hkv, lo_bit = spec["n_hi"], spec["Hkv"], spec["lo_bit"]
    npg = k.shape[0] // 32
    pool = np.zeros(max(npg, 1) * Hkv * oracle.page_bytes(n_hi, lo_bit, spec.get("v_bit", 2)), np.uint8)
    rs = np.zeros((1, Hkv, 128), np.float32)
    rq = np.zeros_like(rs)
    rc = np.zeros((1, Hkv), np.int32)
    st = oracle.quantize_pages(Hkv, n_hi, 1 if running else 0, 1, k, v, np.arange(npg, dtype=np.int32),
                               pool, max(npg, 1), seq_of_page=np.zeros(npg, np.int32), n_seqs=1,
                               run_sum=rs, run_sumsq=rq, run_count=rc, lo_bit=lo_bit,
                               v_bit=spec.get("v_bit", 2))
    assert st == 0
    return pool, (rs, rq, rc)


@pytest.mark.parametrize("name", ["llama3_8b", "qwen3_8b", "long", "budget", "budget_84",
                                  "budget_kv4", "llama3_70b"])
def test_fullsize_sampled(name):
    import torch
    import bench
    from tests.kitty_cases import attn_error
    oracle.set_threads(8)
    spec = bench.workload_spec(name, 8)
    spec["layers"] = 1
    B = spec["B"]
    keep = sorted({0, B // 2, B - 1} | ({int(np.argmax(spec["tails"]))} if B > 1 else set()))
    cfg, layers, raw = bench.build_layers(spec, 8, keep=keep)
    lc = layers[0]
    blob = oracle.page_bytes(spec["n_hi"], spec["lo_bit"], spec.get("v_bit", 2))
    gpool = lc.pool.cpu().numpy()
    bt = lc.block_table.cpu().numpy()      # host-chosen page ids (an input)
    gen = torch.Generator(device="cuda").manual_seed(77)
    q = torch.randn((B, spec["Hq"], 128), generator=gen, device="cuda").to(torch.bfloat16)
    out = torch.empty((B, spec["Hq"], 128), dtype=torch.float32, device="cuda")
    lc.attend(q.view(torch.int16), out, sm_scale=SM)
    torch.cuda.synchronize()
    assert int(lc.status.item()) == 0
    qh = q.view(torch.int16).cpu().numpy().view(np.uint16)
    got_all = out.cpu().numpy().astype(np.float64)
    for b in keep:
        k, v, tk, tv = raw[0][b]
        npg = int(spec["pages"][b])
        opool, _ = _oracle_seq_pool(spec, k, v, spec["running"])
        per_page = blob * spec["Hkv"]
        for p in range(npg):
            pid = bt[b, p]
            assert (gpool[pid * per_page:(pid + 1) * per_page] == opool[p * per_page:(p + 1) * per_page]).all(), \
                "sequence %d page %d differs" % (b, p)
        tl = int(spec["tails"][b])
        ref, st = oracle.decode_attention(
            spec["Hkv"], spec["Hq"], spec["n_hi"], 1, qh[b:b + 1], opool, max(npg, 1),
            np.arange(max(npg, 1), dtype=np.int32)[None, :], np.array([npg], np.int32),
            tk[None], tv[None], np.array([tl], np.int32), SM, lo_bit=spec["lo_bit"],
            v_bit=spec.get("v_bit", 2))
        assert st == 0
        excess, rel = attn_error(got_all[b:b + 1], ref)
        print("%s sequence %d: max |gpu - oracle| = %.3e of RMS" % (name, b, rel))
        assert excess <= 0, "sequence %d: max err %.3e of RMS" % (b, rel)


def test_fullsize_serving_append_steps():
    """The serving workload's append path at full size: 33 steps so every sampled
    sequence flushes once, pages and running statistics bit-exact."""
    import torch
    import bench
    spec = bench.workload_spec("budget", 40)
    spec["layers"] = 1
    B, Hkv = spec["B"], spec["Hkv"]
    keep = [0, int(np.argmax(spec["tails"])), B - 1]
    cfg, layers, raw = bench.build_layers(spec, 40, keep=keep)
    lc = layers[0]
    gen = torch.Generator(device="cuda").manual_seed(5)
    plans = []
    for step in range(33):
        kn = torch.randn((B, Hkv, 128), generator=gen, device="cuda").to(torch.bfloat16).view(torch.int16)
        vn = torch.randn((B, Hkv, 128), generator=gen, device="cuda").to(torch.bfloat16).view(torch.int16)
        fl = lc.plan_flush()
        plans.append((kn.cpu().numpy().view(np.uint16), vn.cpu().numpy().view(np.uint16), fl))
        lc.append(kn, vn, torch.from_numpy(fl).cuda())
    torch.cuda.synchronize()
    assert int(lc.status.item()) == 0
    gpool = lc.pool.cpu().numpy()
    per_page = oracle.page_bytes(spec["n_hi"], spec["lo_bit"], spec.get("v_bit", 2)) * Hkv
    g_sum = lc.run_sum.cpu().numpy()
    g_cnt = lc.run_count.cpu().numpy()
    g_np = lc.num_pages.cpu().numpy()
    g_bt = lc.block_table.cpu().numpy()
    for b in keep:
        k, v, tk, tv = raw[0][b]
        npg = int(spec["pages"][b])
        opool, (rs, rq, rc) = _oracle_seq_pool(spec, k, v, True)
        # continue the oracle sequence with the same tokens and flush ids
        pool_pages = npg + 2
        big = np.zeros(pool_pages * per_page, np.uint8)
        big[:opool.size] = opool
        tail_k, tail_v = tk[None].copy(), tv[None].copy()
        tl = np.array([spec["tails"][b]], np.int32)
        btab = np.full((1, npg + 2), -1, np.int32)
        btab[0, :npg] = np.arange(npg)
        nump = np.array([npg], np.int32)
        flushed = []
        for kn, vn, fl in plans:
            f = np.array([npg + len(flushed) if fl[b] >= 0 else -1], np.int32)
            if fl[b] >= 0:
                flushed.append(int(fl[b]))
            st = oracle.append_token(Hkv, spec["n_hi"], 1, 1, kn[b:b + 1], vn[b:b + 1], tail_k, tail_v, tl,
                                     rs, rq, rc, f, btab, npg + 2, nump, big, pool_pages)
            assert st == 0
        assert flushed, "sampled sequence %d never flushed" % b
        assert g_np[b] == nump[0] and (g_bt[b, npg:nump[0]] == flushed).all()
        for i, pid in enumerate(flushed):
            assert (gpool[pid * per_page:(pid + 1) * per_page] ==
                    big[(npg + i) * per_page:(npg + i + 1) * per_page]).all()
        assert (g_sum[b].view(np.uint32) == rs[0].view(np.uint32)).all()
        assert (g_cnt[b] == rc[0]).all()
