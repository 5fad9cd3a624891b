"""Paged Kitty KV cache state for a decode loop (the runtime around the kernels).

Per layer: a pool of packed pages, a block table, per-sequence unquantized
tails, running channel statistics and a host page allocator.  The host keeps a
mirror of every tail length and page count, so it decides flushes (which
sequences complete a 32-token page this step, and which physical page each one
gets) without reading device memory; the device state is only ever changed by
the library's kernels.  Paper: Abstract (page-centric layout, lightweight
runtime pipeline); VeloxQuant-MLX docs, Decode phase.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

from . import kitty

PAGE = 32
D = 128


class LayerCache:
    def __init__(self, cfg: kitty.Config, B: int, max_pages: int, pool_pages: int,
                 device="cuda"):
        self.cfg, self.B, self.max_pages, self.pool_pages = cfg, B, max_pages, pool_pages
        blob, per_page = kitty.page_bytes(cfg)
        self.blob, self.per_page = blob, per_page
        Hkv = cfg.num_kv_heads
        dev = torch.device(device)
        self.pool = torch.zeros(pool_pages * per_page, dtype=torch.uint8, device=dev)
        self.block_table = torch.full((B, max_pages), -1, dtype=torch.int32, device=dev)
        self.num_pages = torch.zeros(B, dtype=torch.int32, device=dev)
        self.tail_k = torch.zeros((B, Hkv, PAGE, D), dtype=torch.int16, device=dev)
        self.tail_v = torch.zeros_like(self.tail_k)
        self.tail_len = torch.zeros(B, dtype=torch.int32, device=dev)
        running = cfg.rank_mode != kitty.RANK_PAGE  # running or sequence-wide ranking
        self.run_sum = torch.zeros((B, Hkv, D), dtype=torch.float32, device=dev) if running else None
        self.run_sumsq = torch.zeros_like(self.run_sum) if running else None
        self.run_count = torch.zeros((B, Hkv), dtype=torch.int32, device=dev) if running else None
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.alloc = kitty.PageAllocator(pool_pages)
        self.h_tail = np.zeros(B, np.int64)
        self.h_pages = np.zeros(B, np.int64)
        ws = kitty.decode_workspace_bytes(cfg, B, max_pages)
        self.workspace = torch.empty(max(ws, 16) // 4, dtype=torch.float32, device=dev)

    # -- prefill: n_pages[b] full pages and a tail of tails[b] tokens per sequence
    def prefill(self, k_pages, v_pages, n_pages, k_tail=None, v_tail=None, tails=None,
                page_order=None, stream=None):
        """k_pages, v_pages: 16-bit tensors (int16 view) [sum(n_pages)*32, Hkv, D],
        sequence-major; k_tail, v_tail: [B, Hkv, 32, D] with tails[b] valid rows.
        page_order: optional permutation of the allocated ids (shuffled block table)."""
        n_pages = np.asarray(n_pages, np.int64)
        tails = np.zeros(self.B, np.int64) if tails is None else np.asarray(tails, np.int64)
        tot = int(n_pages.sum())
        dev = self.pool.device
        ids = self.alloc.alloc(tot)
        if page_order is not None:
            ids = ids[np.asarray(page_order)]
        bt = np.full((self.B, self.max_pages), -1, np.int32)
        off = 0
        for b in range(self.B):
            bt[b, :n_pages[b]] = ids[off:off + n_pages[b]]
            off += n_pages[b]
        self.block_table.copy_(torch.from_numpy(bt))
        self.num_pages.copy_(torch.from_numpy(n_pages.astype(np.int32)))
        run = {}
        if self.run_sum is not None:
            seq = np.repeat(np.arange(self.B), n_pages).astype(np.int32)
            run = dict(seq_of_page=torch.from_numpy(seq).to(dev), n_seqs=self.B,
                       run_sum=self.run_sum, run_sumsq=self.run_sumsq, run_count=self.run_count)
        if tot:
            kitty.quantize_pages(self.cfg, k_pages, v_pages,
                                 torch.from_numpy(ids.astype(np.int32)).to(dev), self.pool,
                                 self.pool_pages, status=self.status, stream=stream, **run)
        if k_tail is not None:
            self.tail_k.copy_(k_tail)
            self.tail_v.copy_(v_tail)
        self.tail_len.copy_(torch.from_numpy(tails.astype(np.int32)))
        self.h_tail[:] = tails
        self.h_pages[:] = n_pages
        self.set_plan_hint()
        return ids

    def set_plan_hint(self, total_pages=None, max_pages=None):
        """Give the decode split planner the batch's total and largest page counts
        (default: the host mirror's) on this cache's own copy of the config, and
        grow the workspace if that plan needs more.  Any values are correct;
        close ones balance the splits better."""
        total = int(self.h_pages.sum()) if total_pages is None else int(total_pages)
        mx = int(self.h_pages.max()) if max_pages is None and self.B else int(max_pages or 0)
        self.cfg = dataclasses.replace(self.cfg, decode_total_pages=total, decode_max_pages=mx)
        need = kitty.decode_workspace_bytes(self.cfg, self.B, self.max_pages)
        if need > self.workspace.numel() * 4:
            self.workspace = torch.empty(need // 4, dtype=torch.float32, device=self.pool.device)

    def plan_flush(self) -> np.ndarray:
        """Host decision for the next append: a fresh page id for each sequence whose
        tail completes a page, -1 elsewhere; advances the host mirror."""
        fl = np.full(self.B, -1, np.int32)
        full = np.nonzero(self.h_tail + 1 == PAGE)[0]
        full = full[self.h_pages[full] < self.max_pages]
        if full.size:
            fl[full] = self.alloc.alloc(full.size)
        self.h_tail += 1
        self.h_tail[full] = 0
        self.h_pages[full] += 1
        return fl

    def step(self, k_new, v_new, flush_ids, q, out, sm_scale=None, stream=None):
        """append(k_new, v_new, flush_ids) then attend(q, out) as one fused launch
        (plus the split combine).  The fused call takes query groups of at most 4
        heads per kv head; larger groups make the two calls."""
        if self.cfg.num_q_heads // self.cfg.num_kv_heads > 4:
            self.append(k_new, v_new, flush_ids, stream=stream)
            self.attend(q, out, sm_scale, stream=stream)
            return
        sm = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
        kitty.append_decode(self.cfg, k_new, v_new, q, self.tail_k, self.tail_v, self.tail_len,
                            self.run_sum, self.run_sumsq, self.run_count, flush_ids,
                            self.block_table, self.num_pages, self.pool, self.pool_pages, sm, out,
                            workspace=self.workspace, status=self.status, stream=stream)

    def capture_step(self, k_new, v_new, flush_ids, q, out, sm_scale=None):
        """A CUDA graph of one fused step(k_new, v_new, flush_ids, q, out) on these
        tensors: replaying it runs the call on what the tensors hold then, on the
        current stream.  Capturing runs nothing; the cache state changes only on
        replay."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step(k_new, v_new, flush_ids, q, out, sm_scale)
        return g

    def append(self, k_new, v_new, flush_ids, stream=None):
        kitty.append_token(self.cfg, k_new, v_new, self.tail_k, self.tail_v, self.tail_len,
                           self.run_sum, self.run_sumsq, self.run_count, flush_ids,
                           self.block_table, self.num_pages, self.pool, self.pool_pages,
                           status=self.status, stream=stream)

    def attend(self, q, out, sm_scale=None, stream=None):
        sm = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
        kitty.decode_attention(self.cfg, q, self.pool, self.pool_pages, self.block_table,
                               self.num_pages, self.tail_k, self.tail_v, self.tail_len, sm, out,
                               workspace=self.workspace, status=self.status, stream=stream)

    def append_bytes(self, flush_ids, fused: bool = False) -> int:
        """Bytes one append must move: the new K/V token read and written into the
        tail and, per flushed (sequence, kv head), the full tail read, the page blob
        written and the running statistics read and written.  fused: the flushed
        page is attended from on-chip memory, so the read of it that
        algorithmic_bytes counts is taken off here."""
        Hkv = self.cfg.num_kv_heads
        nf = int((np.asarray(flush_ids) >= 0).sum())
        stats = 2 * 2 * D * 4 + 2 * 4 if self.run_sum is not None else 0
        page = PAGE * D * 2 * 2 + self.blob + stats - (self.blob if fused else 0)
        return self.B * Hkv * D * 2 * 2 * 2 + nf * Hkv * page

    def kv_tokens(self) -> int:
        """Cached tokens one decode call attends to, over the batch (host mirror):
        full pages and unquantized tail tokens."""
        return int(self.h_pages.sum()) * PAGE + int(self.h_tail.sum())

    def algorithmic_bytes(self) -> int:
        """Bytes one decode call must move: packed pages + tails + Q + O + block
        table entries (host mirror of the current lengths)."""
        Hkv, Hq = self.cfg.num_kv_heads, self.cfg.num_q_heads
        pages = int(self.h_pages.sum())
        return (pages * Hkv * self.blob + int(self.h_tail.sum()) * Hkv * D * 2 * 2
                + self.B * Hq * D * 2 * 2 + pages * 4)


class F16LayerCache:
    """The unquantized 16-bit paged KV cache of one layer (the paper's comparison
    layout for its same-budget claims, Abstract), with the same decode-loop
    interface as LayerCache: every token lives in a 32-token page (no tail), a
    token that starts a page gets a fresh page id from the host allocator, and
    the host mirrors every length."""

    def __init__(self, cfg: kitty.Config, B: int, max_pages: int, pool_pages: int,
                 device="cuda"):
        self.cfg, self.B, self.max_pages, self.pool_pages = cfg, B, max_pages, pool_pages
        blob, per_page = kitty.f16kv_page_bytes(cfg)
        self.blob, self.per_page = blob, per_page
        dev = torch.device(device)
        self.pool = torch.zeros(pool_pages * per_page, dtype=torch.uint8, device=dev)
        self.block_table = torch.full((B, max_pages), -1, dtype=torch.int32, device=dev)
        self.ctx_len = torch.zeros(B, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.alloc = kitty.PageAllocator(pool_pages)
        self.h_len = np.zeros(B, np.int64)
        ws = kitty.f16kv_workspace_bytes(cfg, B, max_pages)
        self.workspace = torch.empty(max(ws, 16) // 4, dtype=torch.float32, device=dev)

    def prefill(self, k_pages, v_pages, n_pages, k_tail=None, v_tail=None, tails=None,
                page_order=None, stream=None):
        """As LayerCache.prefill: n_pages[b] full pages (k_pages, v_pages 16-bit
        [sum(n_pages)*32, Hkv, D], sequence-major) and tails[b] more tokens
        (k_tail, v_tail [B, Hkv, 32, D]), which go to a last, partial page."""
        n_pages = np.asarray(n_pages, np.int64)
        tails = np.zeros(self.B, np.int64) if tails is None else np.asarray(tails, np.int64)
        tot = int(n_pages.sum())
        dev = self.pool.device
        ids = self.alloc.alloc(tot)
        if page_order is not None:
            ids = ids[np.asarray(page_order)]
        with_tail = np.nonzero(tails > 0)[0]
        tail_ids = self.alloc.alloc(with_tail.size) if with_tail.size else np.zeros(0, np.int32)
        bt = np.full((self.B, self.max_pages), -1, np.int32)
        off = 0
        for b in range(self.B):
            bt[b, :n_pages[b]] = ids[off:off + n_pages[b]]
            off += n_pages[b]
        for i, b in enumerate(with_tail):
            bt[b, n_pages[b]] = tail_ids[i]
        self.block_table.copy_(torch.from_numpy(bt))
        if tot:
            kitty.f16kv_write_pages(self.cfg, k_pages, v_pages,
                                    torch.from_numpy(ids.astype(np.int32)).to(dev), self.pool,
                                    self.pool_pages, status=self.status, stream=stream)
        if with_tail.size:
            sel = torch.from_numpy(with_tail).to(dev)
            kt = k_tail.index_select(0, sel).transpose(1, 2).contiguous()  # [n, 32, Hkv, D]
            vt = v_tail.index_select(0, sel).transpose(1, 2).contiguous()
            kitty.f16kv_write_pages(self.cfg, kt, vt,
                                    torch.from_numpy(tail_ids.astype(np.int32)).to(dev),
                                    self.pool, self.pool_pages, status=self.status, stream=stream)
        self.h_len[:] = n_pages * PAGE + tails
        self.ctx_len.copy_(torch.from_numpy(self.h_len.astype(np.int32)))
        return ids

    def plan_flush(self) -> np.ndarray:
        """Host decision for the next append: a fresh page id for each sequence whose
        next token starts a page, -1 elsewhere; advances the host mirror."""
        fl = np.full(self.B, -1, np.int32)
        new = np.nonzero(self.h_len % PAGE == 0)[0]
        new = new[self.h_len[new] // PAGE < self.max_pages]
        if new.size:
            fl[new] = self.alloc.alloc(new.size)
        self.h_len += 1
        return fl

    def append(self, k_new, v_new, new_page_ids, stream=None):
        kitty.f16kv_append(self.cfg, k_new, v_new, self.pool, self.pool_pages, self.block_table,
                           self.ctx_len, new_page_ids, status=self.status, stream=stream)

    def attend(self, q, out, sm_scale=None, stream=None):
        sm = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
        kitty.f16kv_decode(self.cfg, q, self.pool, self.pool_pages, self.block_table,
                           self.ctx_len, sm, out, workspace=self.workspace, status=self.status,
                           stream=stream)

    def step(self, k_new, v_new, new_page_ids, q, out, sm_scale=None, stream=None):
        """append then attend (the append's two kernels, the decode and its combine)."""
        self.append(k_new, v_new, new_page_ids, stream=stream)
        self.attend(q, out, sm_scale, stream=stream)

    def append_bytes(self, new_page_ids, fused: bool = False) -> int:
        """The new K/V token read and written into its page."""
        return self.B * self.cfg.num_kv_heads * D * 2 * 2 * 2

    def kv_tokens(self) -> int:
        return int(self.h_len.sum())

    def algorithmic_bytes(self) -> int:
        """Bytes one decode call must move: the K and V rows of every cached token,
        Q, O and the block-table entries (host mirror of the lengths)."""
        Hkv, Hq = self.cfg.num_kv_heads, self.cfg.num_q_heads
        pages = int(((self.h_len + PAGE - 1) // PAGE).sum())
        return (int(self.h_len.sum()) * Hkv * D * 2 * 2 + self.B * Hq * D * 2 * 2 + pages * 4)


def capture_layers_step(layers, k_new, v_new, flush_ids, q, out, sm_scale=None,
                        fused: bool = True):
    """One CUDA graph of a decode step over every layer: per layer l in order, the
    fused step(k_new[l], v_new[l], flush_ids[l], q[l], out[l]) (fused=False:
    append then attend).  Each argument is indexed by layer (a list, or a tensor
    with a leading layer dimension).  The layers' kernels run back to back inside
    one graph, so a step costs one graph launch instead of one per layer.
    Capturing runs nothing; replaying runs the calls on what the tensors hold then,
    on the current stream."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for l, lc in enumerate(layers):
            if fused:
                lc.step(k_new[l], v_new[l], flush_ids[l], q[l], out[l], sm_scale)
            else:
                lc.append(k_new[l], v_new[l], flush_ids[l])
                lc.attend(q[l], out[l], sm_scale)
    return g


class ServingStep:
    """One decode step of every layer from pinned host memory, with the copies
    overlapped with the kernels.

    Per layer, the query rows and the new Key/Value token sit in one contiguous
    pinned block (views: q[l], k_new[l], v_new[l]; the caller writes them before
    run()), copied up with one transfer on an upload stream; the layer's call
    waits only for its own block, and its output comes back on a download stream
    while later layers compute.  run() returns once every output is in `out`
    (pinned host, [L][B][Hq][D]).

    graphs=True: the whole step (uploads, every layer's call, downloads) is one
    CUDA graph, so a step costs one graph launch.  The flush ids of the next
    step are planned on the host while the graph of this one runs (the host
    mirrors of the layers run one step ahead between calls); two graphs read
    the plans from alternating pinned buffers.  Between run() calls the layers
    must not be driven by other calls.
    graphs=False: direct calls; the flush plan of layer l is made just before
    its block goes up, so planning overlaps the kernels of the layers before it.
    fused=False runs append then attend per layer.
    """

    def __init__(self, layers, graphs: bool = True, fused: bool = True, sm_scale=None):
        self.layers = layers
        lc0 = layers[0]
        L, B = len(layers), lc0.B
        Hq, Hkv = lc0.cfg.num_q_heads, lc0.cfg.num_kv_heads
        dev = lc0.pool.device
        self.sizes = [B * Hq * D * 2, B * Hkv * D * 2, B * Hkv * D * 2, B * 4]
        per = sum(self.sizes)
        self.block = (per + 255) // 256 * 256  # 256-byte aligned per-layer blocks
        self.h_in = torch.empty(L * self.block, dtype=torch.uint8).pin_memory()
        self.d_in = torch.empty(L * self.block, dtype=torch.uint8, device=dev)
        self.q, self.k_new, self.v_new, self.flush = [], [], [], []
        self._dq, self._dk, self._dv, self._dfl = [], [], [], []
        for l in range(L):
            hv_, dv_ = self._views(self.h_in, l, B, Hq, Hkv), self._views(self.d_in, l, B, Hq, Hkv)
            for lst, x in zip((self.q, self.k_new, self.v_new, self.flush), hv_):
                lst.append(x)
            for lst, x in zip((self._dq, self._dk, self._dv, self._dfl), dv_):
                lst.append(x)
        out_dt = torch.bfloat16 if lc0.cfg.in_dtype == kitty.BF16 else torch.float16
        self.d_out = torch.empty((L, B, Hq, D), dtype=out_dt, device=dev)
        self.out = torch.empty((L, B, Hq, D), dtype=out_dt).pin_memory()
        self.up, self.down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        self.ev_in = [torch.cuda.Event() for _ in range(L)]
        self.ev_out = [torch.cuda.Event() for _ in range(L)]
        self.fused, self.sm_scale = fused, sm_scale
        self.graphs = None
        if graphs:
            # flush plans of two consecutive steps, and their device copy
            self.h_fl = [torch.empty((L, B), dtype=torch.int32).pin_memory() for _ in range(2)]
            self.d_fl = torch.empty((L, B), dtype=torch.int32, device=dev)
            self.graphs = [self._capture(p) for p in range(2)]
            self._parity = 0
            self._planned = 0  # layers whose flushes of the pending step are planned

    def _views(self, buf, l, B, Hq, Hkv):
        o = l * self.block
        s = self.sizes
        q = buf[o:o + s[0]].view(torch.int16).view(B, Hq, D)
        k = buf[o + s[0]:o + s[0] + s[1]].view(torch.int16).view(B, Hkv, D)
        v = buf[o + s[0] + s[1]:o + s[0] + s[1] + s[2]].view(torch.int16).view(B, Hkv, D)
        f = buf[o + s[0] + s[1] + s[2]:o + s[0] + s[1] + s[2] + s[3]].view(torch.int32)
        return q, k, v, f

    def _call(self, l, flush_ids):
        lc = self.layers[l]
        if self.fused:
            lc.step(self._dk[l], self._dv[l], flush_ids, self._dq[l], self.d_out[l], self.sm_scale)
        else:
            lc.append(self._dk[l], self._dv[l], flush_ids)
            lc.attend(self._dq[l], self.d_out[l], self.sm_scale)

    def _capture(self, parity):
        """The graph of one step reading its flush plan from h_fl[parity]."""
        qkv = sum(self.sizes[:3])
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cap = torch.cuda.current_stream()
            self.up.wait_stream(cap)
            self.down.wait_stream(cap)
            with torch.cuda.stream(self.up):
                self.d_fl.copy_(self.h_fl[parity], non_blocking=True)
                for l in range(len(self.layers)):
                    o = l * self.block
                    self.d_in[o:o + qkv].copy_(self.h_in[o:o + qkv], non_blocking=True)
                    self.ev_in[l].record(self.up)
            for l in range(len(self.layers)):
                cap.wait_event(self.ev_in[l])
                self._call(l, self.d_fl[l])
                self.ev_out[l].record(cap)
                with torch.cuda.stream(self.down):
                    self.down.wait_event(self.ev_out[l])
                    self.out[l].copy_(self.d_out[l], non_blocking=True)
            cap.wait_stream(self.down)
        return g

    def _plan(self, parity):
        """Plans the pending step's flushes into h_fl[parity], from the first layer
        not yet planned: a layer whose page allocation fails raises, and the next
        call resumes at that layer."""
        fl = self.h_fl[parity].numpy()
        while self._planned < len(self.layers):
            fl[self._planned] = self.layers[self._planned].plan_flush()
            self._planned += 1

    def bytes_up(self) -> int:
        return len(self.layers) * sum(self.sizes)

    def bytes_down(self) -> int:
        return self.out.numel() * self.out.element_size()

    def run(self):
        cur = torch.cuda.current_stream()
        if self.graphs is not None:
            self._plan(self._parity)  # nothing left to do unless the look-ahead stopped
            self.graphs[self._parity].replay()
            self._parity ^= 1
            self._planned = 0
            try:
                self._plan(self._parity)  # the next step's flushes, while this one runs
            except kitty.KittyError:
                pass  # e.g. the pool is full: raised by the next run(), before its step
            cur.synchronize()
            return self.out
        # the device input blocks and outputs may still be in use by work queued
        # before this call
        self.up.wait_stream(cur)
        self.down.wait_stream(cur)
        for l, lc in enumerate(self.layers):
            self.flush[l].numpy()[:] = lc.plan_flush()
            o = l * self.block
            with torch.cuda.stream(self.up):
                self.d_in[o:o + self.block].copy_(self.h_in[o:o + self.block], non_blocking=True)
                self.ev_in[l].record(self.up)
            cur.wait_event(self.ev_in[l])
            self._call(l, self._dfl[l])
            self.ev_out[l].record(cur)
            with torch.cuda.stream(self.down):
                self.down.wait_event(self.ev_out[l])
                self.out[l].copy_(self.d_out[l], non_blocking=True)
        self.down.synchronize()
        return self.out
