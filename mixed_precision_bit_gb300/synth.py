"""Seeded synthetic workloads for Kitty decode (inputs only, no method arithmetic).

Shapes follow the paper's model families (Llama-3-8B and Qwen3-8B decode layers:
32 query heads, 8 KV heads, head_dim 128).  No dataset or trained weights are
used; the value distributions mimic Key caches with outlier channels:

* Q, V ~ N(0, 1);  K[t, c] = N(0, 1) * sigma[h, c], sigma ~ lognormal(0, 1) drawn
  per KV head and channel (redrawn every ``drift`` tokens for the long-context
  workload, so boosted channel lists differ between pages);
* values rounded once to the input dtype (fp16 or bf16, round-to-nearest-even);
* physical page ids: a Fisher-Yates shuffle of [0, n_pages) (random block table).

Two generators: ``host_*`` uses a counter-based splitmix64 stream in numpy
(bit-reproducible on any machine; used where the oracle sees every input), and
``device_*`` uses a seeded torch generator on the GPU for workloads too large to
build on the host (sampled sequences are copied back for the oracle).
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

D = 128
PAGE = 32
F16, BF16 = 0, 1

_GOLD = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, tag: str) -> np.uint64:
    h = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    for ch in tag.encode():
        with np.errstate(over="ignore"):
            h = _mix(np.asarray([h ^ np.uint64(ch)], np.uint64) + _GOLD)[0]
    return h


def bits(seed: int, tag: str, n: int, start: int = 0) -> np.ndarray:
    """n raw 64-bit draws of the splitmix64 stream (seed, tag), from index start."""
    i = np.arange(start, start + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(_key(seed, tag) + (i + np.uint64(1)) * _GOLD)


def uniform(seed, tag, n, start=0) -> np.ndarray:
    """U[0, 1) with 53-bit resolution."""
    return (bits(seed, tag, n, start) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed, tag, n, start=0) -> np.ndarray:
    """N(0, 1) by the Box-Muller cosine branch over consecutive uniform pairs."""
    u = uniform(seed, tag, 2 * n, 2 * start)
    u1 = 1.0 - u[0::2]
    u2 = u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def to_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round float values to fp16 / bf16 (nearest-even) and return the raw uint16 bits."""
    if dtype == F16:
        return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16)


def from_bits(b: np.ndarray, dtype: int) -> np.ndarray:
    b = np.asarray(b, np.uint16)
    if dtype == F16:
        return b.view(np.float16).astype(np.float32)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def shuffle(seed: int, tag: str, n: int) -> np.ndarray:
    """Fisher-Yates permutation of [0, n) driven by the stream (seed, tag)."""
    perm = np.arange(n, dtype=np.int32)
    r = bits(seed, tag, max(n, 1))
    for i in range(n - 1, 0, -1):
        j = int(r[i] % np.uint64(i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    return perm


@dataclasses.dataclass
class Workload:
    """One decode-layer workload: per-sequence cached lengths and shapes."""
    name: str
    B: int
    Hq: int
    Hkv: int
    n_hi: int
    dtype: int
    pages: np.ndarray      # [B] quantized pages per sequence
    tails: np.ndarray      # [B] unquantized tail tokens (0..31)
    drift: int = 0         # redraw K channel scales every `drift` tokens (0: never)
    layers: int = 1
    lo_bit: int = 2        # Key plane width: 2 ((hi, lo) = (4, 2) bits) or 4 ((8, 4))
    v_bit: int = 2         # Value code width: 2, or 4 (with lo_bit 4)

    @property
    def g(self):
        return self.Hq // self.Hkv

    @property
    def max_pages(self):
        return int(self.pages.max()) if self.B else 0

    @property
    def total_pages(self):
        return int(self.pages.sum())


def workload(name: str, seed: int = 0) -> Workload:
    """The named workloads.

    tiny       1 seq, 1 KV head, 1 query head, 256 tokens (8 pages), fp16, n_hi=32
    llama3_8b  16 seqs, 32/8 heads, bf16, 4096 tokens (128 pages), n_hi=32, no tail
    qwen3_8b   64 seqs, 32/8 heads, bf16, 8192 tokens (256 pages) + tail U{0..31}, n_hi=16
    long       8 seqs, 32/8 heads, bf16, lengths U[16384, 65536], n_hi=32, channel
               scales redrawn every 4096 tokens
    llama3_70b 16 seqs, 64/8 heads (query groups of 8), bf16, 8192 tokens (256
               pages) + tail U{0..31}, n_hi=32
    small_gqa  parity-size GQA case: 3 seqs, 8/2 heads, bf16, ragged lengths
    qwen3_g1, qwen3_g2
               qwen3_8b with 8 / 16 query heads (query groups of 1 and 2): the
               decode kernel's per-page cost does not depend on the group size
    """
    if name == "tiny":
        return Workload(name, 1, 1, 1, 32, F16, np.array([8]), np.array([0]))
    if name == "llama3_8b":
        return Workload(name, 16, 32, 8, 32, BF16, np.full(16, 128), np.zeros(16, np.int64))
    if name in ("qwen3_8b", "qwen3_g1", "qwen3_g2"):
        tails = (bits(seed, "qwen3_8b/tail", 64) % np.uint64(32)).astype(np.int64)
        Hq = {"qwen3_8b": 32, "qwen3_g1": 8, "qwen3_g2": 16}[name]
        return Workload(name, 64, Hq, 8, 16, BF16, np.full(64, 256), tails)
    if name == "long":
        L = 16384 + (bits(seed, "long/len", 8) % np.uint64(65536 - 16384 + 1)).astype(np.int64)
        return Workload(name, 8, 32, 8, 32, BF16, L // PAGE, L % PAGE, drift=4096)
    if name == "llama3_70b":
        tails = (bits(seed, "llama3_70b/tail", 16) % np.uint64(32)).astype(np.int64)
        return Workload(name, 16, 64, 8, 32, BF16, np.full(16, 256), tails)
    if name == "small_gqa":
        return Workload(name, 3, 8, 2, 32, BF16, np.array([5, 0, 9]), np.array([7, 3, 31]))
    raise KeyError(name)


def budget_batch(budget_bytes: int, layers: int, Hkv: int, ctx_pages: int, blob: int,
                 tail_bytes: int, stat_bytes: int) -> int:
    """Largest batch whose pages (+ full tails + running stats) fit the KV budget."""
    per_seq = layers * (Hkv * (ctx_pages + 1) * blob + tail_bytes + stat_bytes)
    return budget_bytes // per_seq


# ------------------------------------------------------------------ host inputs
def host_inputs(w: Workload, seed: int = 0):
    """All inputs of a workload as numpy arrays (small and medium workloads).

    Returns dict with k, v: uint16 [total_pages*32, Hkv, D] (sequence-major page
    order), page_ids / seq_of_page [total_pages], block_table [B, max_pages],
    num_pages [B], tail_k / tail_v [B, Hkv, 32, D], tail_len [B], q [B, Hq, D],
    pool_pages.
    """
    ntok_seq = w.pages * PAGE + w.tails
    tok_k, tok_v = [], []
    for b in range(w.B):
        n = int(ntok_seq[b])
        z = normal(seed, "k/%d" % b, n * w.Hkv * D).reshape(n, w.Hkv, D)
        vv = normal(seed, "v/%d" % b, n * w.Hkv * D).reshape(n, w.Hkv, D)
        seg = np.arange(n) // w.drift if w.drift else np.zeros(n, np.int64)
        for s in np.unique(seg):
            sig = np.exp(normal(seed, "sigma/%d" % s, w.Hkv * D)).reshape(w.Hkv, D)
            z[seg == s] *= sig
        tok_k.append(to_bits(z, w.dtype))
        tok_v.append(to_bits(vv, w.dtype))
    return _assemble(w, seed, tok_k, tok_v,
                     to_bits(normal(seed, "q", w.B * w.Hq * D).reshape(w.B, w.Hq, D), w.dtype))


def _assemble(w, seed, tok_k, tok_v, q):
    tot = w.total_pages
    k = np.zeros((tot * PAGE, w.Hkv, D), np.uint16)
    v = np.zeros_like(k)
    tail_k = np.zeros((w.B, w.Hkv, PAGE, D), np.uint16)
    tail_v = np.zeros_like(tail_k)
    ids = shuffle(seed, "page_ids", tot)
    mp = max(w.max_pages, 1)
    block_table = np.full((w.B, mp), -1, np.int32)
    seq_of_page = np.zeros(tot, np.int32)
    off = 0
    for b in range(w.B):
        npg, tl = int(w.pages[b]), int(w.tails[b])
        k[off * PAGE:(off + npg) * PAGE] = tok_k[b][:npg * PAGE]
        v[off * PAGE:(off + npg) * PAGE] = tok_v[b][:npg * PAGE]
        tail_k[b, :, :tl] = tok_k[b][npg * PAGE:].transpose(1, 0, 2)
        tail_v[b, :, :tl] = tok_v[b][npg * PAGE:].transpose(1, 0, 2)
        block_table[b, :npg] = ids[off:off + npg]
        seq_of_page[off:off + npg] = b
        off += npg
    return dict(k=k, v=v, page_ids=ids.astype(np.int32), seq_of_page=seq_of_page,
                block_table=block_table, num_pages=w.pages.astype(np.int32),
                tail_k=tail_k, tail_v=tail_v, tail_len=w.tails.astype(np.int32), q=q,
                pool_pages=max(tot, 1))


# ------------------------------------------------------------------ device inputs
def device_kv(w: Workload, b: int, seed: int, device, n_tok=None):
    """K, V (torch, input dtype) [n_tok, Hkv, D] of sequence b, generated on `device`
    from a seeded torch generator; the same call on the host device gives the same
    draws only up to the generator's platform behaviour, so callers copy device
    tensors back when the oracle needs them."""
    import torch
    n = int(w.pages[b] * PAGE + w.tails[b]) if n_tok is None else n_tok
    dt = torch.float16 if w.dtype == F16 else torch.bfloat16
    gen = torch.Generator(device=device)
    gen.manual_seed((seed * 1000003 + b * 7919 + 17) & 0x7FFFFFFFFFFFFFFF)
    z = torch.randn((n, w.Hkv, D), generator=gen, device=device, dtype=torch.float32)
    vv = torch.randn((n, w.Hkv, D), generator=gen, device=device, dtype=torch.float32)
    sg = torch.Generator(device=device)
    nseg = (n + w.drift - 1) // w.drift if w.drift else 1
    for s in range(max(nseg, 1)):
        sg.manual_seed((seed * 1000003 + 99991 * (s + 1)) & 0x7FFFFFFFFFFFFFFF)
        sig = torch.exp(torch.randn((w.Hkv, D), generator=sg, device=device))
        lo = s * w.drift if w.drift else 0
        hi = min(n, (s + 1) * w.drift) if w.drift else n
        z[lo:hi] *= sig
    return z.to(dt), vv.to(dt)


def host_fast_normal(seed: int, shape) -> np.ndarray:
    """N(0, 1) from numpy's seeded PCG64 (fast bulk draws for CPU timing samples,
    where bit-reproducibility across the two paths is not needed)."""
    return np.random.default_rng(seed).standard_normal(shape, dtype=np.float32)
