"""ctypes binding of libkitty.so (C ABI in include/kitty.h).

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors are torch tensors on the GPU (their data pointers are passed through);
the stream defaults to torch's current stream.  There is no fallback: if the
library cannot be built or loaded, the calls raise.
"""

from __future__ import annotations

import ctypes
import dataclasses
import os

from . import build as _build

OK = 0
ERR = {-1: "KITTY_ERR_INVALID_ARG", -2: "KITTY_ERR_UNSUPPORTED", -3: "KITTY_ERR_CUDA",
       -4: "KITTY_ERR_WORKSPACE", -5: "KITTY_ERR_OOM"}
ST = dict(OK=0, EMPTY=1, RANGE=2, NONFINITE=3, BAD_PAGE=4, BAD_LEN=5, TAIL_FULL=6,
          BAD_FLUSH=7, TABLE_FULL=8, BAD_SEQ=9, TIMEOUT=10)
F16, BF16, F32 = 0, 1, 2
RANK_PAGE, RANK_RUNNING, RANK_SEQUENCE = 0, 1, 2


class KittyError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__("%s returned %s (%d)" % (fn, ERR.get(code, "?"), code))
        self.code = code


class _Cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "head_dim", "num_kv_heads", "num_q_heads", "page_tokens", "n_hi", "hi_bit", "lo_bit",
        "v_group", "rank_mode", "in_dtype", "decode_pages_per_split", "decode_total_pages",
        "decode_max_pages", "decode_wait_polls", "v_bit")]


@dataclasses.dataclass
class Config:
    num_kv_heads: int
    num_q_heads: int
    n_hi: int = 32
    in_dtype: int = BF16
    rank_mode: int = RANK_PAGE
    decode_pages_per_split: int = 0
    decode_total_pages: int = 0     # planning hint: the batch's total page count (0: unknown)
    decode_max_pages: int = 0       # planning hint: the longest sequence's page count (0: unknown)
    decode_wait_polls: int = 0      # bound of the decode page waits in polls (0: the library's)
    head_dim: int = 128
    page_tokens: int = 32
    hi_bit: int = 4
    lo_bit: int = 2
    v_group: int = 32
    v_bit: int = 2                  # Value code width: 2, or 4 with lo_bit 4

    def c(self):
        return _Cfg(self.head_dim, self.num_kv_heads, self.num_q_heads, self.page_tokens,
                    self.n_hi, self.hi_bit, self.lo_bit, self.v_group, self.rank_mode,
                    self.in_dtype, self.decode_pages_per_split, self.decode_total_pages,
                    self.decode_max_pages, self.decode_wait_polls, self.v_bit)


_lib = None
EXPORTS = ("kitty_abi_version", "kitty_page_bytes", "kitty_avg_bits", "kitty_alloc_create",
           "kitty_alloc_pages", "kitty_free_pages", "kitty_alloc_free_count",
           "kitty_alloc_destroy", "kitty_quantize_pages", "kitty_append_token",
           "kitty_decode_workspace_bytes", "kitty_decode_attention", "kitty_decode_plan",
           "kitty_decode_attention_noalloc", "kitty_append_decode", "kitty_f16kv_page_bytes",
           "kitty_f16kv_write_pages", "kitty_f16kv_append", "kitty_f16kv_workspace_bytes",
           "kitty_f16kv_decode")
NOALLOC_SCRATCH_BYTES = 8 << 20


def lib_path() -> str:
    return _build.LIB


def load():
    """Load libkitty.so, building it first if it is missing or stale."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        C = ctypes.POINTER(_Cfg)
        sig = {
            "kitty_abi_version": (ctypes.c_int, []),
            "kitty_page_bytes": (ctypes.c_int, [C, ctypes.POINTER(sz), ctypes.POINTER(sz)]),
            "kitty_avg_bits": (ctypes.c_float, [C]),
            "kitty_alloc_create": (ctypes.c_int, [i32, ctypes.POINTER(P)]),
            "kitty_alloc_pages": (ctypes.c_int, [P, i32, P]),
            "kitty_free_pages": (ctypes.c_int, [P, i32, P]),
            "kitty_alloc_free_count": (i32, [P]),
            "kitty_alloc_destroy": (None, [P]),
            "kitty_quantize_pages": (ctypes.c_int, [C, P, P, i32, P, P, i32, P, P, P, P, i32, P, P]),
            "kitty_append_token": (ctypes.c_int, [C, P, P, P, P, P, P, P, P, P, P, i32, P, P, i32,
                                                  i32, P, P]),
            "kitty_decode_workspace_bytes": (ctypes.c_int, [C, i32, i32, ctypes.POINTER(sz)]),
            "kitty_decode_attention": (ctypes.c_int, [C, P, P, i32, P, i32, P, P, P, P,
                                                      ctypes.c_float, P, i32, P, sz, i32, P, P]),
            "kitty_decode_attention_noalloc": (ctypes.c_int, [C, P, P, i32, P, i32, P, P, P, P,
                                                              ctypes.c_float, P, i32, i32, P, P]),
            "kitty_append_decode": (ctypes.c_int, [C, P, P, P, P, P, P, P, P, P, P, P, i32, P, P, i32,
                                                   ctypes.c_float, P, i32, P, sz, i32, P, P]),
            "kitty_decode_plan": (ctypes.c_int, [C, i32, i32, ctypes.POINTER(i32),
                                                 ctypes.POINTER(i32)]),
            "kitty_f16kv_page_bytes": (ctypes.c_int, [C, ctypes.POINTER(sz), ctypes.POINTER(sz)]),
            "kitty_f16kv_write_pages": (ctypes.c_int, [C, P, P, i32, P, P, i32, P, P]),
            "kitty_f16kv_append": (ctypes.c_int, [C, P, P, P, i32, P, i32, P, P, i32, P, P]),
            "kitty_f16kv_workspace_bytes": (ctypes.c_int, [C, i32, i32, ctypes.POINTER(sz)]),
            "kitty_f16kv_decode": (ctypes.c_int, [C, P, P, i32, P, i32, P, ctypes.c_float, P, i32,
                                                  P, sz, i32, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _chk(name, rc):
    if rc != OK:
        raise KittyError(name, rc)


def _ptr(t):
    """Device address of a tensor argument.  The library reads and writes plain
    dense arrays in device memory, so a view with gaps or a host tensor is
    refused here (it would be read wrongly, or fault)."""
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_cuda:
        raise ValueError("kitty: tensor arguments must be in device memory (got %s)" % t.device)
    if not t.is_contiguous():
        raise ValueError("kitty: tensor arguments must be contiguous (shape %s, strides %s)"
                         % (tuple(t.shape), t.stride()))
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def page_bytes(cfg: Config):
    b, p = ctypes.c_size_t(), ctypes.c_size_t()
    _chk("kitty_page_bytes", load().kitty_page_bytes(ctypes.byref(cfg.c()), ctypes.byref(b),
                                                     ctypes.byref(p)))
    return b.value, p.value


def avg_bits(cfg: Config) -> float:
    return float(load().kitty_avg_bits(ctypes.byref(cfg.c())))


class PageAllocator:
    """Host free list of physical page ids (kitty_alloc_*)."""

    def __init__(self, num_pages: int):
        h = ctypes.c_void_p()
        _chk("kitty_alloc_create", load().kitty_alloc_create(num_pages, ctypes.byref(h)))
        self._h = h

    def alloc(self, n: int):
        import numpy as np
        out = np.zeros(n, np.int32)
        _chk("kitty_alloc_pages", load().kitty_alloc_pages(self._h, n, out.ctypes.data))
        return out

    def free(self, ids):
        import numpy as np
        ids = np.ascontiguousarray(ids, np.int32)
        _chk("kitty_free_pages", load().kitty_free_pages(self._h, ids.size, ids.ctypes.data))

    @property
    def free_count(self) -> int:
        return int(load().kitty_alloc_free_count(self._h))

    def close(self):
        if self._h:
            load().kitty_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def quantize_pages(cfg: Config, k, v, page_ids, pool, pool_pages: int, seq_of_page=None,
                   n_seqs: int = 0, run_sum=None, run_sumsq=None, run_count=None, status=None,
                   stream=None):
    n_pages = page_ids.numel()
    _chk("kitty_quantize_pages", load().kitty_quantize_pages(
        ctypes.byref(cfg.c()), _ptr(k), _ptr(v), n_pages, _ptr(page_ids), _ptr(seq_of_page),
        n_seqs, _ptr(run_sum), _ptr(run_sumsq), _ptr(run_count), _ptr(pool), pool_pages,
        _ptr(status), _stream(stream)))


def append_token(cfg: Config, k_new, v_new, tail_k, tail_v, tail_len, run_sum, run_sumsq,
                 run_count, flush_page_ids, block_table, num_pages, pool, pool_pages: int,
                 status=None, stream=None):
    B = tail_len.numel()
    _chk("kitty_append_token", load().kitty_append_token(
        ctypes.byref(cfg.c()), _ptr(k_new), _ptr(v_new), _ptr(tail_k), _ptr(tail_v),
        _ptr(tail_len), _ptr(run_sum), _ptr(run_sumsq), _ptr(run_count), _ptr(flush_page_ids),
        _ptr(block_table), block_table.shape[1], _ptr(num_pages), _ptr(pool), pool_pages, B,
        _ptr(status), _stream(stream)))


def decode_workspace_bytes(cfg: Config, B: int, max_pages: int) -> int:
    n = ctypes.c_size_t()
    _chk("kitty_decode_workspace_bytes", load().kitty_decode_workspace_bytes(
        ctypes.byref(cfg.c()), B, max_pages, ctypes.byref(n)))
    return n.value


def decode_plan(cfg: Config, B: int, max_pages: int):
    s, c = ctypes.c_int32(), ctypes.c_int32()
    _chk("kitty_decode_plan", load().kitty_decode_plan(ctypes.byref(cfg.c()), B, max_pages,
                                                       ctypes.byref(s), ctypes.byref(c)))
    return s.value, c.value


def decode_attention(cfg: Config, q, pool, pool_pages: int, block_table, num_pages, tail_k,
                     tail_v, tail_len, sm_scale: float, out, workspace=None, status=None,
                     stream=None, out_dtype=None):
    import torch
    B = num_pages.numel()
    if out_dtype is None:
        out_dtype = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}[out.dtype]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _chk("kitty_decode_attention", load().kitty_decode_attention(
        ctypes.byref(cfg.c()), _ptr(q), _ptr(pool), pool_pages, _ptr(block_table),
        block_table.shape[1], _ptr(num_pages), _ptr(tail_k), _ptr(tail_v), _ptr(tail_len),
        float(sm_scale), _ptr(out), out_dtype, _ptr(workspace), ws_bytes, B, _ptr(status),
        _stream(stream)))


def decode_attention_noalloc(cfg: Config, q, pool, pool_pages: int, block_table, num_pages,
                             tail_k, tail_v, tail_len, sm_scale: float, out, status=None,
                             stream=None, out_dtype=None):
    """kitty_decode_attention without a workspace: the library keeps the split-K
    partials in its own fixed device array (no allocation during the call)."""
    import torch
    B = num_pages.numel()
    if out_dtype is None:
        out_dtype = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}[out.dtype]
    _chk("kitty_decode_attention_noalloc", load().kitty_decode_attention_noalloc(
        ctypes.byref(cfg.c()), _ptr(q), _ptr(pool), pool_pages, _ptr(block_table),
        block_table.shape[1], _ptr(num_pages), _ptr(tail_k), _ptr(tail_v), _ptr(tail_len),
        float(sm_scale), _ptr(out), out_dtype, B, _ptr(status), _stream(stream)))


def append_decode(cfg: Config, k_new, v_new, q, tail_k, tail_v, tail_len, run_sum, run_sumsq,
                  run_count, flush_page_ids, block_table, num_pages, pool, pool_pages: int,
                  sm_scale: float, out, workspace=None, status=None, stream=None, out_dtype=None):
    """append_token followed by decode_attention, as one fused launch."""
    import torch
    B = tail_len.numel()
    if out_dtype is None:
        out_dtype = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}[out.dtype]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _chk("kitty_append_decode", load().kitty_append_decode(
        ctypes.byref(cfg.c()), _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(tail_k), _ptr(tail_v),
        _ptr(tail_len), _ptr(run_sum), _ptr(run_sumsq), _ptr(run_count), _ptr(flush_page_ids),
        _ptr(block_table), block_table.shape[1], _ptr(num_pages), _ptr(pool), pool_pages,
        float(sm_scale), _ptr(out), out_dtype, _ptr(workspace), ws_bytes, B, _ptr(status),
        _stream(stream)))


# ------------------------------------------------------------------ 16-bit paged baseline
def f16kv_page_bytes(cfg: Config):
    b, p = ctypes.c_size_t(), ctypes.c_size_t()
    _chk("kitty_f16kv_page_bytes", load().kitty_f16kv_page_bytes(
        ctypes.byref(cfg.c()), ctypes.byref(b), ctypes.byref(p)))
    return b.value, p.value


def f16kv_write_pages(cfg: Config, k, v, page_ids, pool, pool_pages: int, status=None,
                      stream=None):
    _chk("kitty_f16kv_write_pages", load().kitty_f16kv_write_pages(
        ctypes.byref(cfg.c()), _ptr(k), _ptr(v), page_ids.numel(), _ptr(page_ids), _ptr(pool),
        pool_pages, _ptr(status), _stream(stream)))


def f16kv_append(cfg: Config, k_new, v_new, pool, pool_pages: int, block_table, ctx_len,
                 new_page_ids, status=None, stream=None):
    _chk("kitty_f16kv_append", load().kitty_f16kv_append(
        ctypes.byref(cfg.c()), _ptr(k_new), _ptr(v_new), _ptr(pool), pool_pages,
        _ptr(block_table), block_table.shape[1], _ptr(ctx_len), _ptr(new_page_ids),
        ctx_len.numel(), _ptr(status), _stream(stream)))


def f16kv_workspace_bytes(cfg: Config, B: int, max_pages: int) -> int:
    n = ctypes.c_size_t()
    _chk("kitty_f16kv_workspace_bytes", load().kitty_f16kv_workspace_bytes(
        ctypes.byref(cfg.c()), B, max_pages, ctypes.byref(n)))
    return n.value


def f16kv_decode(cfg: Config, q, pool, pool_pages: int, block_table, ctx_len, sm_scale: float,
                 out, workspace=None, status=None, stream=None, out_dtype=None):
    import torch
    B = ctx_len.numel()
    if out_dtype is None:
        out_dtype = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}[out.dtype]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _chk("kitty_f16kv_decode", load().kitty_f16kv_decode(
        ctypes.byref(cfg.c()), _ptr(q), _ptr(pool), pool_pages, _ptr(block_table),
        block_table.shape[1], _ptr(ctx_len), float(sm_scale), _ptr(out), out_dtype,
        _ptr(workspace), ws_bytes, B, _ptr(status), _stream(stream)))
