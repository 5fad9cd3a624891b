"""GPU check of the pipelined multi-layer serving step (cache.ServingStep), and
of the one-graph step over every layer (cache.capture_layers_step).

Its copies run on side streams, overlapped with the kernels. Over many decode
steps with page flushes, it must give outputs and cache state bit-identical to
the same per-layer calls made directly on the same inputs: the fused call
(LayerCache.step), or append then attend. Those calls themselves are checked
against the oracle in test_gpu_fused.py and test_gpu_parity.py."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixed_precision_bit_gb300 import kitty
    kitty.load()


def _layers(L, B, Hkv, Hq, n_hi, pages, tails, gen):
    import torch
    from mixed_precision_bit_gb300 import kitty
    from mixed_precision_bit_gb300.cache import LayerCache
    cfg = kitty.Config(num_kv_heads=Hkv, num_q_heads=Hq, n_hi=n_hi, in_dtype=kitty.BF16,
                       rank_mode=kitty.RANK_RUNNING)
    max_pages = int(max(pages)) + 4
    pool_pages = int(sum(pages)) + B * 4
    out = []
    for _ in range(L):
        lc = LayerCache(cfg, B, max_pages, pool_pages)
        tot = int(sum(pages))
        kp = (torch.randn((tot * 32, Hkv, 128), generator=gen, device="cuda") *
              torch.exp(torch.randn((1, Hkv, 128), generator=gen, device="cuda")))
        vp = torch.randn((tot * 32, Hkv, 128), generator=gen, device="cuda")
        kt = torch.randn((B, Hkv, 32, 128), generator=gen, device="cuda")
        vt = torch.randn((B, Hkv, 32, 128), generator=gen, device="cuda")
        bf = lambda x: x.to(torch.bfloat16).view(torch.int16)
        lc.prefill(bf(kp), bf(vp), pages, bf(kt), bf(vt), tails)
        out.append(lc)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("graphs,fused,Hq", [(True, True, 8), (False, True, 8), (True, False, 8),
                                             (True, True, 16)],
                         ids=["graphs", "direct", "graphs-unfused", "graphs-g8"])
def test_serving_step_matches_per_layer_calls(graphs, fused, Hq):
    """Hq = 16 (query groups of 8): the step makes the append and the decode as
    two calls, and must equal them made directly."""
    import torch
    from mixed_precision_bit_gb300.cache import ServingStep
    L, B, Hkv, n_hi = 3, 5, 2, 32
    pages, tails = [3, 1, 0, 2, 4], [30, 31, 5, 0, 17]
    ref = _layers(L, B, Hkv, Hq, n_hi, pages, tails, torch.Generator("cuda").manual_seed(3))
    new = _layers(L, B, Hkv, Hq, n_hi, pages, tails, torch.Generator("cuda").manual_seed(3))
    # a first plain call outside any graph capture
    q0 = torch.zeros((B, Hq, 128), dtype=torch.int16, device="cuda")
    o0 = torch.empty((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    new[0].attend(q0, o0)
    torch.cuda.synchronize()
    srv = ServingStep(new, graphs=graphs, fused=fused)
    g = torch.Generator("cuda").manual_seed(5)
    d_out = torch.empty((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    flushes = 0
    for step in range(40):
        q = torch.randn((L, B, Hq, 128), generator=g, device="cuda").to(torch.bfloat16).view(torch.int16)
        k = torch.randn((L, B, Hkv, 128), generator=g, device="cuda").to(torch.bfloat16).view(torch.int16)
        v = torch.randn((L, B, Hkv, 128), generator=g, device="cuda").to(torch.bfloat16).view(torch.int16)
        for l in range(L):
            srv.q[l].copy_(q[l].cpu())
            srv.k_new[l].copy_(k[l].cpu())
            srv.v_new[l].copy_(v[l].cpu())
        got = srv.run().clone()
        for l, lc in enumerate(ref):
            fl = lc.plan_flush()
            flushes += int((fl >= 0).sum())
            fd = torch.from_numpy(fl).cuda()
            if fused and Hq // Hkv <= 4:
                lc.step(k[l], v[l], fd, q[l], d_out)
            else:  # the same two calls (the fused call attends a flushed page in another order)
                lc.append(k[l], v[l], fd)
                lc.attend(q[l], d_out)
            want = d_out.cpu()
            assert torch.equal(got[l].view(torch.int16), want.view(torch.int16)), (step, l)
    assert flushes >= 2 * L  # the steps crossed page boundaries
    torch.cuda.synchronize()
    for a, b in zip(ref, new):
        for name in ("pool", "block_table", "num_pages", "tail_k", "tail_v", "tail_len",
                     "run_sum", "run_sumsq", "run_count", "status"):
            assert torch.equal(getattr(a, name), getattr(b, name)), name
        assert int(b.status.item()) == 0
    assert srv.bytes_up() == L * (B * Hq * 128 * 2 + 2 * B * Hkv * 128 * 2 + B * 4)


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "unfused"])
def test_layers_step_graph_matches_per_layer_calls(fused):
    """One graph over every layer's call of a step (capture_layers_step), replayed
    on new inputs each step, against the same calls made directly: outputs and
    cache state bit-identical, across page flushes."""
    import torch
    from mixed_precision_bit_gb300.cache import capture_layers_step
    L, B, Hkv, Hq, n_hi = 3, 5, 2, 8, 32
    pages, tails = [3, 1, 0, 2, 4], [30, 31, 5, 0, 17]
    ref = _layers(L, B, Hkv, Hq, n_hi, pages, tails, torch.Generator("cuda").manual_seed(3))
    new = _layers(L, B, Hkv, Hq, n_hi, pages, tails, torch.Generator("cuda").manual_seed(3))
    q_in = torch.empty((L, B, Hq, 128), dtype=torch.int16, device="cuda")
    k_in = torch.empty((L, B, Hkv, 128), dtype=torch.int16, device="cuda")
    v_in = torch.empty_like(k_in)
    fl_in = torch.full((L, B), -1, dtype=torch.int32, device="cuda")
    out = torch.empty((L, B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    graph = capture_layers_step(new, k_in, v_in, fl_in, q_in, out, fused=fused)
    g = torch.Generator("cuda").manual_seed(5)
    d_out = torch.empty((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    flushes = 0
    for step in range(40):
        q = torch.randn((L, B, Hq, 128), generator=g, device="cuda").to(torch.bfloat16).view(torch.int16)
        k = torch.randn((L, B, Hkv, 128), generator=g, device="cuda").to(torch.bfloat16).view(torch.int16)
        v = torch.randn((L, B, Hkv, 128), generator=g, device="cuda").to(torch.bfloat16).view(torch.int16)
        plans = [lc.plan_flush() for lc in new]
        q_in.copy_(q)
        k_in.copy_(k)
        v_in.copy_(v)
        fl_in.copy_(torch.from_numpy(np.stack(plans)))
        graph.replay()
        for l, lc in enumerate(ref):
            fl = lc.plan_flush()
            assert (fl == plans[l]).all()
            flushes += int((fl >= 0).sum())
            fd = torch.from_numpy(fl).cuda()
            if fused:
                lc.step(k[l], v[l], fd, q[l], d_out)
            else:
                lc.append(k[l], v[l], fd)
                lc.attend(q[l], d_out)
            assert torch.equal(out[l].view(torch.int16), d_out.view(torch.int16)), (step, l)
    assert flushes >= 2 * L
    torch.cuda.synchronize()
    for a, b in zip(ref, new):
        for name in ("pool", "block_table", "num_pages", "tail_k", "tail_v", "tail_len",
                     "run_sum", "run_sumsq", "run_count", "status"):
            assert torch.equal(getattr(a, name), getattr(b, name)), name
        assert int(b.status.item()) == 0


_FRESH = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
from mixed_precision_bit_gb300 import kitty
from mixed_precision_bit_gb300.cache import LayerCache
cfg = kitty.Config(num_kv_heads=2, num_q_heads=8, n_hi=32, in_dtype=kitty.BF16,
                   rank_mode=kitty.RANK_RUNNING)
g = torch.Generator("cuda").manual_seed(1)
bf = lambda *s: torch.randn(s, generator=g, device="cuda").to(torch.bfloat16).view(torch.int16)
caches = []
for _ in range(2):
    lc = LayerCache(cfg, 3, 8, 32)
    g.manual_seed(2)
    lc.prefill(bf(3 * 32, 2, 128), bf(3 * 32, 2, 128), [1, 2, 0], bf(3, 2, 32, 128), bf(3, 2, 32, 128), [5, 31, 0])
    caches.append(lc)
torch.cuda.synchronize()
q, k, v = bf(3, 8, 128), bf(3, 2, 128), bf(3, 2, 128)
fl = torch.full((3,), -1, dtype=torch.int32, device="cuda")
o1 = torch.empty((3, 8, 128), dtype=torch.bfloat16, device="cuda")
o2 = torch.empty_like(o1)
graph = caches[0].capture_step(k, v, fl, q, o1)   # the first decode launch of this process
graph.replay()
caches[1].step(k, v, fl, q, o2)
torch.cuda.synchronize()
assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
assert int(caches[0].status.item()) == 0
print("ok")
"""


def test_capture_as_first_call_in_a_fresh_process():
    """A graph captured before any plain call (a new CUDA context: the library's
    first launch happens inside the capture) replays like a plain call."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH, root], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
