#!/usr/bin/env python
"""Kitty decode-step benchmark on GB300.

Default workload ("budget"): a fixed 40 GB KV budget of Kitty pages (n_hi=32,
2.5-bit Keys) holding Llama-3-8B-shaped layers (32 query / 8 KV heads,
head_dim 128, 32 layers), context 8192 tokens (256 pages) + an unquantized tail
of U{0..31} tokens per sequence, batch maximised for the budget.  One step =
for every layer: append one token per sequence (running sum/sum-of-squares
statistics, flushing tails that complete a 32-token page into a freshly
allocated page) and split-K paged decode attention over the layer's cache.
Metric: decode tokens/s = sequences x steps / time; HBM GB/s of the decode
kernel on algorithmic bytes (packed pages + tails + Q + O + block table).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kitty|reference]
                       [--workload budget|budget_uniform|budget_k4|budget_84|budget_kv4|budget_fp16|
                                   llama3_8b|llama3_70b|qwen3_8b|qwen3_g1|qwen3_g2|long|tiny]
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn tokens/s & HBM GB/s (% of 8 TB/s) over Kitty 2-bit paged KV, 1 GB300"
NOMINAL_HBM_GBS = 8000.0
PAGE, D = 32, 128


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# ------------------------------------------------------------------ workloads
def workload_spec(name: str, steps_total: int):
    """Shapes of the benchmark workloads (one GPU)."""
    import numpy as np
    from mixed_precision_bit_gb300 import synth
    if name == "budget_fp16":
        # the unquantized 16-bit paged layout on the same 40 GB budget (16 KB per
        # (page, kv head), no tail or statistics): the comparison layout of the
        # paper's batch and throughput claims
        Hkv, Hq, layers, ctx_pages = 8, 32, 32, 256
        B = synth.budget_batch(40 * 10 ** 9, layers, Hkv, ctx_pages, 2 * PAGE * D * 2, 0, 0)
        tails = (synth.bits(0, "budget/tail", B) % np.uint64(32)).astype(np.int64)
        return dict(name=name, B=int(B), Hq=Hq, Hkv=Hkv, n_hi=0, layers=layers, running=False,
                    pages=np.full(B, ctx_pages, np.int64), tails=tails, drift=0,
                    budget_bytes=40 * 10 ** 9, dtype=synth.BF16, lo_bit=2, f16kv=True)
    if name in ("budget", "budget_uniform", "budget_k4", "budget_84", "budget_kv4"):
        # budget: Kitty (top 32 of 128 Key channels at 4 bits, running statistics);
        # budget_uniform: every Key channel at 2 bits; budget_k4: every Key channel
        # at 4 bits (n_hi = 128, two 2-bit planes); budget_84: Kitty at (8, 4) bits
        # (top 32 channels at 8 bits, the rest at 4, two 4-bit planes, running
        # statistics).  Values are 2-bit in these four.  budget_kv4: uniform 4-bit
        # KV (every Key channel at 4 bits in one 4-bit plane, 4-bit Values).
        n_hi = {"budget": 32, "budget_uniform": 0, "budget_k4": 128, "budget_84": 32,
                "budget_kv4": 0}[name]
        lo_bit = 4 if name in ("budget_84", "budget_kv4") else 2
        v_bit = 4 if name == "budget_kv4" else 2
        running = name in ("budget", "budget_84")
        blob = 512 * lo_bit + 4 * lo_bit * n_hi + n_hi + 512 * v_bit + 1024
        Hkv, Hq, layers, ctx_pages = 8, 32, 32, 256
        stat = Hkv * D * 2 * 4 + Hkv * 4 if running else 0
        tail_bytes = 2 * Hkv * PAGE * D * 2
        B = synth.budget_batch(40 * 10 ** 9, layers, Hkv, ctx_pages, blob, tail_bytes, stat)
        tails = (synth.bits(0, "budget/tail", B) % np.uint64(32)).astype(np.int64)
        return dict(name=name, B=int(B), Hq=Hq, Hkv=Hkv, n_hi=n_hi, layers=layers,
                    running=running, pages=np.full(B, ctx_pages, np.int64), tails=tails,
                    drift=0, budget_bytes=40 * 10 ** 9, dtype=synth.BF16, lo_bit=lo_bit,
                    v_bit=v_bit)
    w = synth.workload(name)
    # independent layer copies, rotated every step, so the working set exceeds 4x L2
    pool = w.total_pages * w.Hkv * (512 * w.lo_bit + 4 * w.lo_bit * w.n_hi + w.n_hi
                                    + 512 * w.v_bit + 1024)
    # (the tiny single-head case is latency-bound and stays L2-resident by design)
    layers = 1 if name == "tiny" else max(1, math.ceil(4 * 129e6 / max(pool, 1)))
    return dict(name=name, B=w.B, Hq=w.Hq, Hkv=w.Hkv, n_hi=w.n_hi, layers=layers, running=False,
                pages=w.pages.astype(np.int64), tails=w.tails.astype(np.int64), drift=w.drift,
                budget_bytes=None, dtype=w.dtype, lo_bit=w.lo_bit, v_bit=w.v_bit)


def headroom_pages(tails, steps_total):
    return int(((int(tails.max()) if len(tails) else 0) + steps_total) // PAGE + 1)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region.

    start() waits for the first sample before the region opens and stamps the
    region's start; stop() stamps its end and keeps the samples taken inside
    it.  A region shorter than the 50 ms period keeps the first sample taken
    after it began ("window" says which)."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None
        self.t0 = self.t1 = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def start(self):
        """Waits (at most 5 s) for the first sample, then stamps the region start."""
        if self.p is not None:
            t = time.time()
            while time.time() - t < 5.0 and os.path.getsize(self.f.name) == 0:
                time.sleep(0.01)
        self.t0 = time.time()

    def _rows(self):
        import datetime
        out = []
        self.f.flush()
        self.f.seek(0)
        for line in self.f.read().splitlines():
            r = [x.strip() for x in line.split(", ")]
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                out.append((ts, float(r[2]), float(r[3]), r[6:10]))
            except (ValueError, IndexError):
                continue
        return out

    def stop(self):
        self.t1 = time.time()
        if self.p is None:
            return None
        time.sleep(0.06)   # one more period: the sample that covers the region's end
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        rows = self._rows()
        os.unlink(self.f.name)
        t0 = self.t0 if self.t0 is not None else -1.0
        inside = [r for r in rows if t0 <= r[0] <= self.t1]
        window = "samples inside the timed region"
        if not inside:
            inside = [r for r in rows if r[0] >= t0][:1]
            window = "first sample after the timed region began (region shorter than the period)"
        if not inside:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names, r[3]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median([r[1] for r in inside]),
                "sm_max_mhz": max(r[2] for r in inside), "samples": len(inside),
                "reasons": sorted(reasons), "window": window}


# ------------------------------------------------------------------ kitty arm
def build_layers(spec, steps_total, seed=0, keep=(), pages_per_split=0):
    """Per-layer caches filled with seeded synthetic K/V (generated on the GPU).
    keep: sequences whose raw inputs are copied back to the host (for sampled
    oracle checks); returned as raw[layer][b] = (k, v, tail_k, tail_v) uint16."""
    import numpy as np
    import torch
    from mixed_precision_bit_gb300 import kitty
    from mixed_precision_bit_gb300.cache import F16LayerCache, LayerCache
    Cache = F16LayerCache if spec.get("f16kv") else LayerCache
    B, Hkv, L = spec["B"], spec["Hkv"], spec["layers"]
    pages, tails = spec["pages"], spec["tails"]
    head = headroom_pages(tails, steps_total)
    max_pages = int(pages.max()) + head
    pool_pages = int(pages.sum()) + B * head
    cfg = kitty.Config(num_kv_heads=Hkv, num_q_heads=spec["Hq"], n_hi=spec["n_hi"],
                       in_dtype=spec["dtype"], hi_bit=2 * spec["lo_bit"], lo_bit=spec["lo_bit"],
                       v_bit=spec.get("v_bit", 2),
                       rank_mode=kitty.RANK_RUNNING if spec["running"] else kitty.RANK_PAGE,
                       decode_pages_per_split=pages_per_split)
    tdt = torch.float16 if spec["dtype"] == kitty.F16 else torch.bfloat16
    gen = torch.Generator(device="cuda")
    layers, raw = [], []
    tot = int(pages.sum())
    starts = np.concatenate([[0], np.cumsum(pages)[:-1]]) * PAGE
    for l in range(L):
        lc = Cache(cfg, B, max_pages, pool_pages)
        gen.manual_seed(seed * 7919 + l)
        sig = torch.exp(torch.randn((Hkv, D), generator=gen, device="cuda"))
        kp = torch.empty((tot * PAGE, Hkv, D), dtype=tdt, device="cuda")
        vp = torch.empty_like(kp)
        pos = None
        if spec["drift"]:
            pos = torch.from_numpy(np.concatenate([np.arange(int(p) * PAGE) for p in pages])).cuda()
        chunk = 1 << 20
        for s0 in range(0, tot * PAGE, chunk):
            n = min(chunk, tot * PAGE - s0)
            z = torch.randn((n, Hkv, D), generator=gen, device="cuda")
            if pos is not None:
                seg = pos[s0:s0 + n] // spec["drift"]
                gs = torch.Generator(device="cuda")
                for sgi in torch.unique(seg).tolist():
                    gs.manual_seed(seed * 104729 + 31 * sgi + 1)
                    sg = torch.exp(torch.randn((Hkv, D), generator=gs, device="cuda"))
                    m = seg == sgi
                    z[m] = z[m] * sg
            else:
                z = z * sig
            kp[s0:s0 + n] = z.to(tdt)
            vp[s0:s0 + n] = torch.randn((n, Hkv, D), generator=gen, device="cuda").to(tdt)
        tk = (torch.randn((B, Hkv, PAGE, D), generator=gen, device="cuda") * sig[None, :, None, :]
              ).to(tdt)
        tv = torch.randn((B, Hkv, PAGE, D), generator=gen, device="cuda").to(tdt)
        order = torch.randperm(tot, generator=torch.Generator().manual_seed(seed * 31 + l)).numpy()
        lc.prefill(kp.view(torch.int16), vp.view(torch.int16), pages, tk.view(torch.int16),
                   tv.view(torch.int16), tails, page_order=order)
        host = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
        raw.append({b: (host(kp[starts[b]:starts[b] + pages[b] * PAGE]),
                        host(vp[starts[b]:starts[b] + pages[b] * PAGE]), host(tk[b]), host(tv[b]))
                    for b in keep})
        del kp, vp
        layers.append(lc)
    torch.cuda.synchronize()
    if keep:
        return cfg, layers, raw
    return cfg, layers


def measure_quantize(spec, reps=5, seed=3):
    """Bulk page quantization throughput on one layer of the workload (inputs
    resident): page mode and running mode, timed with CUDA events.  GB/s counts
    the bf16 K+V read plus the packed pages written."""
    import numpy as np
    import torch
    from mixed_precision_bit_gb300 import kitty
    B, Hkv = spec["B"], spec["Hkv"]
    pages = spec["pages"]
    tot = int(pages.sum())
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    tdt = torch.float16 if spec["dtype"] == kitty.F16 else torch.bfloat16
    k = (torch.randn((tot * PAGE, Hkv, D), generator=g, device="cuda")
         * torch.exp(torch.randn((Hkv, D), generator=g, device="cuda"))).to(tdt)
    v = torch.randn((tot * PAGE, Hkv, D), generator=g, device="cuda").to(tdt)
    ids = torch.from_numpy(np.random.default_rng(seed).permutation(tot).astype(np.int32)).cuda()
    seq = torch.from_numpy(np.repeat(np.arange(B), pages).astype(np.int32)).cuda()
    out = {}
    for mode in (kitty.RANK_PAGE, kitty.RANK_RUNNING):
        cfg = kitty.Config(num_kv_heads=Hkv, num_q_heads=spec["Hq"], n_hi=spec["n_hi"],
                           in_dtype=spec["dtype"], rank_mode=mode, hi_bit=2 * spec["lo_bit"],
                           lo_bit=spec["lo_bit"], v_bit=spec.get("v_bit", 2))
        blob, per_page = kitty.page_bytes(cfg)
        pool = torch.empty(tot * per_page, dtype=torch.uint8, device="cuda")
        run = {}
        if mode == kitty.RANK_RUNNING:
            run = dict(seq_of_page=seq, n_seqs=B,
                       run_sum=torch.zeros((B, Hkv, D), dtype=torch.float32, device="cuda"),
                       run_sumsq=torch.zeros((B, Hkv, D), dtype=torch.float32, device="cuda"),
                       run_count=torch.zeros((B, Hkv), dtype=torch.int32, device="cuda"))
        call = lambda: kitty.quantize_pages(cfg, k.view(torch.int16), v.view(torch.int16), ids, pool,
                                            tot, **run)
        call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            call()
        e1.record()
        torch.cuda.synchronize()
        sec = e0.elapsed_time(e1) / 1e3 / reps
        nbytes = 2 * k.numel() * 2 + tot * per_page
        out["page_mode" if mode == kitty.RANK_PAGE else "running_mode"] = {
            "gbs": nbytes / sec / 1e9, "ms": sec * 1e3, "page_heads_per_s": tot * Hkv / sec}
    del k, v
    torch.cuda.empty_cache()
    out["unit"] = "GB/s (bf16 K+V read + packed pages written), one layer of the workload"
    return out


def token_inputs(spec, nsets, seed=1):
    """Per-step new tokens and queries for every layer: nsets distinct sets."""
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    L, B, Hq, Hkv = spec["layers"], spec["B"], spec["Hq"], spec["Hkv"]
    tdt = torch.float16 if spec["dtype"] == 0 else torch.bfloat16
    mk = lambda H: torch.randn((nsets, L, B, H, D), generator=g, device="cuda").to(
        tdt).view(torch.int16)
    return mk(Hq), mk(Hkv), mk(Hkv)


def device_run(args, spec, K, W, steps_total, world, rank, local_rank):
    """Builds the workload's layers, then times K steps (after W warm-up steps) of
    one fused append + decode call per layer, replayed as one CUDA graph per
    step (or as direct calls), with CUDA events on the launching stream and the
    clocks sampled over the timed region."""
    import numpy as np
    import torch
    from mixed_precision_bit_gb300 import kitty
    L, B, Hq = spec["layers"], spec["B"], spec["Hq"]
    # the fused append + decode takes query groups of at most 4
    fused = bool(args.fused) and Hq // spec["Hkv"] <= 4
    cfg, layers = build_layers(spec, steps_total, pages_per_split=args.pages_per_split)
    nsets = max(1, min(4, W))  # every input set's graph is replayed (uploaded) in warm-up
    q_all, kn_all, vn_all = token_inputs(spec, nsets)
    out = torch.empty((L, B, Hq, D), dtype=torch.bfloat16 if spec["dtype"] else torch.float16,
                      device="cuda")
    # flush plans for the warm-up and timed steps, decided on the host ahead of time
    plans, algo, kvtok = [], [], []
    for s in range(W + K):
        plans.append(np.stack([lc.plan_flush() for lc in layers]))
        kvtok.append([lc.kv_tokens() for lc in layers])  # tokens each layer's call attends to
        # bytes of the timed call: the decode call, or the fused append + decode
        # (with graphs, a layer's call is timed with its append also when unfused)
        algo.append([lc.algorithmic_bytes() + (lc.append_bytes(plans[-1][l], fused=fused)
                                               if fused or args.graphs else 0)
                     for l, lc in enumerate(layers)])
    fl_dev = torch.from_numpy(np.stack(plans)).cuda()
    splits, chunk = ((0, 0) if spec.get("f16kv")
                     else kitty.decode_plan(layers[0].cfg, B, layers[0].max_pages))
    stream = torch.cuda.current_stream()
    # CUDA graphs: per input set, one graph of the whole step (every layer's
    # call, in layer order); the step's flush ids are copied into one fixed
    # buffer first.  Without graphs the calls are made directly, with events
    # around each layer's decode call.
    fl_st = torch.full((L, B), -1, dtype=torch.int32, device="cuda")
    graphs = None
    if args.graphs:
        from mixed_precision_bit_gb300.cache import capture_layers_step
        graphs = [capture_layers_step(layers, kn_all[st], vn_all[st], fl_st, q_all[st], out,
                                      fused=fused) for st in range(nsets)]

    def step(s, events):
        st = s % nsets
        if graphs:
            fl_st.copy_(fl_dev[s])
            graphs[st].replay()
            return
        for l, lc in enumerate(layers):
            if not fused:
                lc.append(kn_all[st, l], vn_all[st, l], fl_dev[s, l])
            events[l][0].record(stream)
            if fused:
                lc.step(kn_all[st, l], vn_all[st, l], fl_dev[s, l], q_all[st, l], out[l])
            else:
                lc.attend(q_all[st, l], out[l])
            events[l][1].record(stream)

    ev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
           for _ in range(L)] for _ in range(W + K)]
    for s in range(W):
        step(s, ev[s])
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank) if rank == 0 else None
    if clocks:
        clocks.start()
    t0.record(stream)
    for s in range(K):
        step(W + s, ev[W + s])
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if clocks else None
    ms = dist_max(t0.elapsed_time(t1), world)
    if graphs:
        # one graph per step: a layer's call is timed as the step's time over
        # its layers (an upper bound: the gaps between layers count against it)
        dec_ms = [ms / (K * L)] * (K * L)
    else:
        dec_ms = [ev[W + s][l][0].elapsed_time(ev[W + s][l][1])
                  for s in range(K) for l in range(L)]
    status = [int(lc.status.item()) for lc in layers]
    bad = [x for x in status if x not in (0,)]
    if bad:
        raise RuntimeError("device status codes %s" % bad)
    return dict(cfg=cfg, layers=layers, graphs=graphs, q_all=q_all, kn_all=kn_all, vn_all=vn_all,
                ms=ms, dec_ms=dec_ms,
                dec_bytes=[algo[W + s][l] for s in range(K) for l in range(L)],
                dec_tokens=[kvtok[W + s][l] for s in range(K) for l in range(L)],
                clocks=clk, splits=splits, chunk=chunk, fused=fused)


def target_measure(name, args, world, rank, local_rank, K=200, W=3):
    """The decode call of one single-layer workload (Qwen3-8B-shaped layer,
    long-context layer), timed in the same run as the headline: its call time,
    algorithmic bytes and GB/s against 8 TB/s and the measured copy peak, with
    its own clock samples."""
    import torch
    spec = workload_spec(name, W + K + 2)
    r = device_run(args, spec, K, W, W + K + 2, world, rank, local_rank)
    dec_s = statistics.mean(r["dec_ms"]) / 1e3
    nbytes = statistics.mean(r["dec_bytes"])
    gbs = nbytes / dec_s / 1e9
    peak = float(measured_peaks()[0]["hbm_gbs"])
    res = {"workload": name, "batch": spec["B"], "layers": spec["layers"], "n_hi": spec["n_hi"],
           "context_pages_max": int(spec["pages"].max()), "splits": r["splits"],
           "pages_per_split": r["chunk"], "steps": K, "warmup": W,
           "call_us": dec_s * 1e6, "algorithmic_bytes_per_call": nbytes, "gbs": gbs,
           "pct_of_8tbs": 100.0 * gbs / NOMINAL_HBM_GBS, "pct_of_measured": 100.0 * gbs / peak,
           "decode_tokens_per_s_per_layer": spec["B"] / dec_s,
           "kv_tokens_per_s": sum(r["dec_tokens"]) / (sum(r["dec_ms"]) / 1e3),
           "clocks": r["clocks"]}
    del r
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_kitty(args, rank, world, local_rank):
    import torch
    from mixed_precision_bit_gb300 import kitty
    torch.cuda.set_device(local_rank)
    kitty.load()
    K, W = args.steps, args.warmup
    E = max(1, min(K, args.e2e_steps))
    steps_total = W + K + E + 3   # + two untimed end-to-end steps, + the plan made one step ahead
    spec = workload_spec(args.workload, steps_total)
    if args.layers:
        spec["layers"] = args.layers
    L, B = spec["layers"], spec["B"]
    r0 = device_run(args, spec, K, W, steps_total, world, rank, local_rank)
    layers, graphs = r0["layers"], r0["graphs"]
    cfg, ms, clk, splits, chunk = r0["cfg"], r0["ms"], r0["clocks"], r0["splits"], r0["chunk"]
    q_all, kn_all, vn_all = r0["q_all"], r0["kn_all"], r0["vn_all"]
    dec_ms, dec_bytes, dec_tokens = r0["dec_ms"], r0["dec_bytes"], r0["dec_tokens"]

    # ---- end to end through the public API: host inputs in, outputs back out.
    # ServingStep copies each layer's inputs up and its output back on side
    # streams, overlapped with the other layers' kernels.
    from mixed_precision_bit_gb300.cache import ServingStep
    fused = r0["fused"]
    srv = ServingStep(layers, graphs=bool(args.graphs), fused=fused)
    for l in range(L):
        srv.q[l].copy_(q_all[0, l].cpu())
        srv.k_new[l].copy_(kn_all[0, l].cpu())
        srv.v_new[l].copy_(vn_all[0, l].cpu())
    for _ in range(2):   # untimed: the first replay of each freshly captured graph uploads it
        srv.run()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    w0 = time.perf_counter()
    for s in range(E):
        srv.run()
    e2e_s = dist_max(time.perf_counter() - w0, world)
    status = [int(lc.status.item()) for lc in layers]
    if any(status):
        raise RuntimeError("device status codes after e2e %s" % status)
    h2d = srv.bytes_up()
    d2h = srv.bytes_down()
    launches_per_call = 1 + (1 if splits > 1 else 0)
    pool_bytes = sum(lc.pool.numel() for lc in layers)
    max_pages = layers[0].max_pages
    del srv, layers, graphs, r0, q_all, kn_all, vn_all
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    quant = measure_quantize(spec) if args.measure_quantize and not spec.get("f16kv") else None
    targets = {}
    for name in [t for t in args.targets.split(",") if t]:
        targets[name] = target_measure(name, args, world, rank, local_rank)
    return dict(targets=targets, spec=spec, cfg=cfg, ms=ms, K=K, W=W, E=E, dec_ms=dec_ms, dec_bytes=dec_bytes,
                dec_tokens=dec_tokens,
                quantize=quant,
                clocks=clk, e2e_s=e2e_s, h2d=h2d, d2h=d2h, splits=splits, chunk=chunk,
                gpu_launches=K * L * (2 if fused else 2 + launches_per_call),
                max_pages=max_pages, pool_bytes=pool_bytes, fused=fused)


# ------------------------------------------------------------------ oracle (CPU) arm
def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleSample:
    """A bounded sample of the workload for the CPU oracle: S sequences of one
    layer, quantized by the oracle; one step = append one token per sequence
    (flush where the tail fills) + fp64 decode attention for every head."""

    def __init__(self, spec, S, seed=5):
        import numpy as np
        import oracle
        from mixed_precision_bit_gb300 import synth
        self.o, self.spec = oracle, spec
        self.S = S = min(S, spec["B"])
        Hkv, Hq, n_hi = spec["Hkv"], spec["Hq"], spec["n_hi"]
        pages = spec["pages"][:S]
        tails = spec["tails"][:S].astype(np.int32)
        tot = int(pages.sum())
        self.mode = 1 if spec["running"] else 0
        sig = np.exp(synth.host_fast_normal(seed, (Hkv, D)))
        k = synth.to_bits(synth.host_fast_normal(seed + 1, (tot * PAGE, Hkv, D)) * sig, spec["dtype"])
        v = synth.to_bits(synth.host_fast_normal(seed + 2, (tot * PAGE, Hkv, D)), spec["dtype"])
        self.max_pages = int(pages.max()) + 4
        self.pool_pages = tot + 4 * S
        self.fmt = dict(lo_bit=spec["lo_bit"], v_bit=spec.get("v_bit", 2))
        self.pool = np.zeros(self.pool_pages * Hkv * oracle.page_bytes(n_hi, **self.fmt), np.uint8)
        ids = np.arange(tot, dtype=np.int32)
        self.bt = np.full((S, self.max_pages), -1, np.int32)
        off = 0
        for b in range(S):
            self.bt[b, :pages[b]] = ids[off:off + pages[b]]
            off += pages[b]
        self.rs = np.zeros((S, Hkv, D), np.float32)
        self.rq = np.zeros_like(self.rs)
        self.rc = np.zeros((S, Hkv), np.int32)
        oracle.set_threads(host_cores())
        st = oracle.quantize_pages(Hkv, n_hi, self.mode, spec["dtype"], k, v, ids, self.pool,
                                   self.pool_pages, seq_of_page=np.repeat(np.arange(S), pages),
                                   n_seqs=S, run_sum=self.rs, run_sumsq=self.rq, run_count=self.rc,
                                   **self.fmt)
        assert st == 0, st
        self.tk = synth.to_bits(synth.host_fast_normal(seed + 3, (S, Hkv, PAGE, D)), spec["dtype"])
        self.tv = synth.to_bits(synth.host_fast_normal(seed + 4, (S, Hkv, PAGE, D)), spec["dtype"])
        self.tl = tails.copy()
        self.np_ = pages.astype(np.int32).copy()
        self.q = synth.to_bits(synth.host_fast_normal(seed + 5, (S, Hq, D)), spec["dtype"])
        self.kn = synth.to_bits(synth.host_fast_normal(seed + 6, (S, Hkv, D)), spec["dtype"])
        self.next_id = tot

    def step(self):
        import numpy as np
        from mixed_precision_bit_gb300 import synth
        spec = self.spec
        fl = np.full(self.S, -1, np.int32)
        for b in range(self.S):
            if self.tl[b] + 1 == PAGE and self.np_[b] < self.max_pages and self.next_id < self.pool_pages:
                fl[b] = self.next_id
                self.next_id += 1
        st = self.o.append_token(spec["Hkv"], spec["n_hi"], self.mode, spec["dtype"], self.kn, self.kn,
                                 self.tk, self.tv, self.tl, self.rs, self.rq, self.rc, fl, self.bt,
                                 self.max_pages, self.np_, self.pool, self.pool_pages, **self.fmt)
        _, st2 = self.o.decode_attention(spec["Hkv"], spec["Hq"], spec["n_hi"], spec["dtype"], self.q,
                                         self.pool, self.pool_pages, self.bt, self.np_, self.tk,
                                         self.tv, self.tl, 1.0 / math.sqrt(D), **self.fmt)
        assert st in (0,) and st2 in (0,), (st, st2)


def oracle_tokens_per_s(sample, steps, layers):
    """Times `steps` oracle steps; returns (tokens/s extrapolated to all layers, s/step)."""
    t = []
    for _ in range(steps):
        t0 = time.perf_counter()
        sample.step()
        t.append(time.perf_counter() - t0)
    per = statistics.mean(t)
    return sample.S / (per * layers), per


# ------------------------------------------------------------------ profiled traffic
def kernel_source_digest():
    """sha256 (first 16 hex digits) of the decode kernel's sources with comments
    and blank lines removed: a comment edit keeps a profile's counters valid,
    any code change invalidates them."""
    import hashlib
    import re
    parts = []
    for f in ("decode.cu", "kitty_common.cuh", "quant_tile.cuh"):
        src = open(os.path.join(ROOT, "mixed_precision_bit_gb300", "csrc", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        parts.append("\n".join(l.rstrip() for l in src.splitlines() if l.strip()))
    return hashlib.sha256("\n".join(parts).encode()).hexdigest()[:16]


def profiled_traffic_ratio():
    """DRAM traffic / algorithmic bytes of one decode launch, from the committed ncu
    summary, if that capture was taken on the current kernel source; else None."""
    import re
    path = os.path.join(ROOT, "profiles", "decode_kernel_budget_layer.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = dict(re.findall(r"^\s*(\w+) = (\w+)\s*$", text, re.M))
    if vals.get("kernel_source_sha256_16") != kernel_source_digest():
        return None
    return float(vals["traffic_bytes_per_launch"]) / float(vals["algorithmic_bytes_per_launch"])


# ------------------------------------------------------------------ multi-rank helpers
def dist_max(x: float, world: int) -> float:
    """Max of a per-rank scalar over all ranks (replicas are timed independently;
    the slowest rank defines the job time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, seqs_per_rank: int, steps: int, max_seconds: float) -> float:
    """Whole-job decode tokens/s for replicas: every rank decodes seqs_per_rank
    sequences per step, the job takes the slowest rank's time."""
    return world * seqs_per_rank * steps / max_seconds


# ------------------------------------------------------------------ JSON
def config_block(spec, extra=None):
    c = {"workload": spec["name"],
         "description": ("fixed 40 GB KV budget, Llama-3-8B-shaped layers, context 8192 + tail U{0..31}, "
                         "batch maximised" if spec["budget_bytes"] else "single decode layer"),
         "batch": spec["B"], "layers": spec["layers"], "q_heads": spec["Hq"], "kv_heads": spec["Hkv"],
         "head_dim": D, "page_tokens": PAGE, "n_hi": spec["n_hi"],
         "key_bits": "(hi, lo) = (%d, %d)" % (2 * spec["lo_bit"], spec["lo_bit"]),
         "value_bits": spec.get("v_bit", 2) if not spec.get("f16kv") else 16,
         "rank_mode": "running" if spec["running"] else "page",
         "context_pages": int(spec["pages"].max()), "kv_budget_bytes": spec["budget_bytes"],
         "l2": ("L2-resident (latency-bound tiny case, no roofline claim)" if spec["name"] == "tiny"
                else "inputs larger than L2: %d layer pools rotate every step, > 4x the 129 MB L2"
                % spec["layers"])}
    if extra:
        c.update(extra)
    return c


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kitty", choices=["kitty", "reference"])
    ap.add_argument("--workload", default="budget",
                    choices=["budget", "budget_uniform", "budget_k4", "budget_84", "budget_kv4",
                             "budget_fp16", "llama3_8b", "llama3_70b", "qwen3_8b", "qwen3_g1",
                             "qwen3_g2", "long", "tiny"])
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling)")
    ap.add_argument("--pages-per-split", type=int, default=0,
                    help="decode split-K chunk in pages (0: the library's choice)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--fused", type=int, default=1,
                    help="one fused append + decode call per layer (0: append, then decode)")
    ap.add_argument("--graphs", type=int, default=1,
                    help="replay each layer's append and decode call as CUDA graphs (0: direct calls)")
    ap.add_argument("--cpu-sample", type=int, default=16, help="sequences in the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--measure-quantize", type=int, default=1,
                    help="also time bulk page quantization on one layer (1/0)")
    ap.add_argument("--targets", default="long,qwen3_8b",
                    help="single-layer workloads whose decode call is also timed in this run "
                         "(comma-separated; empty: none)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    peaks, peak_src = measured_peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        spec = workload_spec(args.workload, args.warmup + args.steps)
        sample = OracleSample(spec, args.cpu_sample)
        for _ in range(args.warmup):
            sample.step()
        val, per = oracle_tokens_per_s(sample, args.steps, spec["layers"])
        cores = host_cores()
        desc = "%d of %d sequences, 1 of %d layers (x%d extrapolated), fp64 oracle" % (
            sample.S, spec["B"], spec["layers"], spec["layers"])
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per * 1e3 * spec["layers"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(spec, {"parallelism": "oracle on host cores"}),
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
        return

    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    r = run_kitty(args, rank, world, local_rank)
    spec = r["spec"]
    B, L, K = spec["B"], spec["layers"], r["K"]
    value = job_throughput(world, B, K, r["ms"] / 1e3)
    dec_s = statistics.mean(r["dec_ms"]) / 1e3
    dec_bytes = statistics.mean(r["dec_bytes"])
    achieved = dec_bytes / dec_s / 1e9
    hbm_peak = float(peaks["hbm_gbs"])
    traffic_ratio = profiled_traffic_ratio()
    step_bytes = sum(r["dec_bytes"]) / K
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": r["W"], "ms_per_step": r["ms"] / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "arithmetic": ("bf16 inputs; 2-bit codes as exact fp16 tensor-core operands against fp16 "
                       "hi/lo pairs of the folded scales; fp32 accumulation and online softmax"),
        "data": "synthetic (seeded, on device): K ~ N(0,1)*lognormal channel scales, V,Q ~ N(0,1), bf16",
        "config": config_block(spec, {"parallelism": "replicas" if world > 1 else "single GPU",
                                      "splits": r["splits"], "pages_per_split": r["chunk"],
                                      "pool_bytes": r["pool_bytes"],
                                      "launch": ("fused append + decode per layer" if r["fused"]
                                                 else "append, then decode, per layer") +
                                                (", one CUDA graph per step" if args.graphs else ", direct calls")}),
        "kv_tokens_per_s": sum(r["dec_tokens"]) / (sum(r["dec_ms"]) / 1e3),
        "hbm_gbs": {"decode_kernel": achieved,
                    "step_average": world * step_bytes * K / (r["ms"] / 1e3) / 1e9 / world,
                    "pct_of_8tbs": 100.0 * achieved / NOMINAL_HBM_GBS,
                    "pct_of_measured": 100.0 * achieved / hbm_peak},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak,
                     "traffic": (traffic_ratio * dec_bytes
                                 if traffic_ratio is not None and spec["name"] == "budget" else None),
                     "kernel": ("kitty_append_decode (decode_kernel with the append fused in + "
                                "split combine)" if r["fused"] else
                                "kitty_append_token + kitty_decode_attention" if args.graphs else
                                "kitty_decode_attention (decode_kernel + split combine)"),
                     "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_src,
                     "algorithmic_bytes_per_launch": dec_bytes,
                     "avg_launch_ms": dec_s * 1e3,
                     "launch_timing": ("timed step / layers (one CUDA graph per step)" if args.graphs
                                       else "CUDA events around each call")},
        "gpu_launches": r["gpu_launches"],
        "quantize": r["quantize"],
        "targets": r["targets"],
        "clocks": r["clocks"],
        "e2e": {"value": job_throughput(world, B, r["E"], r["e2e_s"]), "unit": "tokens/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
    }
    if spec.get("f16kv"):
        line["roofline"]["kernel"] = ("kitty_f16kv_append + kitty_f16kv_decode (16-bit paged "
                                      "baseline: decode kernel + split combine)")
        line["config"]["key_bits"] = "16 (unquantized bf16 K and V)"
        line["gpu_launches"] = K * L * 4
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not spec.get("f16kv"):
        sample = OracleSample(spec, args.cpu_sample)
        sample.step()
        steps = 1
        t0 = time.perf_counter()
        vals = []
        while True:
            v, per = oracle_tokens_per_s(sample, 1, L)
            vals.append(per)
            if time.perf_counter() - t0 > 10.0 or len(vals) >= 20:
                break
        per = statistics.mean(vals)
        line["cpu_baseline"] = {
            "value": sample.S / (per * L), "unit": "tokens/s", "cores": host_cores(),
            "kind": "oracle",
            "sample": "%d of %d sequences, 1 of %d layers (x%d extrapolated), %d steps, fp64 oracle"
                      % (sample.S, B, L, L, len(vals))}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
