"""Kitty CPU oracle -- TEST INFRASTRUCTURE ONLY.

ctypes wrapper around ``kitty_oracle.cpp`` (plain C++17, fp32 steps in IEEE
round-to-nearest-even order with no fused multiply-add, fp64 attention).  Only
the tests, the package smoke check and the bench's CPU-baseline leg may import
this module; the library path never does.

Page format, readings and sources are documented in ``kitty_oracle.cpp``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kitty_oracle.cpp")
_OUT = os.path.join(_HERE, "_build", "libkitty_oracle.so")

ST = dict(OK=0, EMPTY=1, RANGE=2, NONFINITE=3, BAD_PAGE=4, BAD_LEN=5, TAIL_FULL=6,
          BAD_FLUSH=7, TABLE_FULL=8, BAD_SEQ=9)


def build(force: bool = False) -> str:
    """Compile the oracle shared library (g++, -O2 -ffp-contract=off)."""
    if not force and os.path.exists(_OUT) and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC):
        return _OUT
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    tmp = _OUT + ".tmp%d" % os.getpid()
    subprocess.check_call(["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                           "-pthread", _SRC, "-o", tmp])
    os.replace(tmp, _OUT)
    return _OUT


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i, f, d = ctypes.c_int, ctypes.c_float, ctypes.c_double
        sig = {
            "orc_abi_version": (i, []),
            "orc_set_threads": (None, [i]),
            "orc_page_bytes": (ctypes.c_long, [i, i, i]),
            "orc_avg_bits": (d, [d, i, i]),
            "orc_f32_to_f16": (ctypes.c_uint16, [f]),
            "orc_step_f16": (ctypes.c_uint16, [f]),
            "orc_f16_to_f32": (f, [ctypes.c_uint16]),
            "orc_bf16_to_f32": (f, [ctypes.c_uint16]),
            "orc_tree_sum": (f, [P]),
            "orc_variance": (f, [f, f, f]),
            "orc_top_k": (None, [P, i, P]),
            "orc_key_pos": (None, [i, i, i, P, P]),
            "orc_key_pos4": (None, [i, i, i, P, P]),
            "orc_val_pos": (None, [i, i, P, P]),
            "orc_val_pos4": (None, [i, i, P, P]),
            "orc_quantize_page_f32": (i, [P, P, i, i, P, P, P, P, i, i]),
            "orc_dequant_page": (None, [P, i, P, P, P, i, i]),
            "orc_page_channels": (None, [P, i, P, i]),
            "orc_meta_pos": (None, [i, i, i, P]),
            "orc_quantize_pages": (i, [i, i, i, i, P, P, i, P, P, i, P, P, P, P, i, i, i]),
            "orc_append_token": (i, [i, i, i, i, P, P, P, P, P, P, P, P, P, P, i, P, P, i, i, i, i]),
            "orc_decode_attention": (i, [i, i, i, i, P, P, i, P, i, P, P, P, P, f, i, P, i, i]),
            "orc_decode_attention_one": (i, [i, i, i, i, P, P, i, P, i, P, P, P, P, f, i, i, P, i, i]),
            "orc_decode_f16kv": (i, [i, i, i, P, P, i, P, i, P, f, i, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dt):
    a = np.ascontiguousarray(a, dtype=dt)
    return a


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def page_bytes(n_hi: int, lo_bit: int = 2, v_bit: int = 2) -> int:
    """Bytes of one (page, kv-head) blob; lo_bit = Key plane width (2: (4, 2)
    configuration, 4: (8, 4)), v_bit = Value code width (2, or 4 with lo_bit 4)."""
    return int(lib().orc_page_bytes(n_hi, lo_bit, v_bit))


def avg_bits(hf: float, hi_bit: int, lo_bit: int) -> float:
    return float(lib().orc_avg_bits(hf, hi_bit, lo_bit))


def f32_to_f16_bits(x: float) -> int:
    return int(lib().orc_f32_to_f16(float(x)))


def step_f16(s: float) -> int:
    """fp16 bits of the stored quantization step for the exact step s >= 0."""
    return int(lib().orc_step_f16(float(s)))


def f16_bits_to_f32(h: int) -> float:
    return float(lib().orc_f16_to_f32(int(h)))


def bf16_bits_to_f32(h: int) -> float:
    return float(lib().orc_bf16_to_f32(int(h)))


def tree_sum(x) -> np.float32:
    x = _c(x, np.float32)
    assert x.size == 32
    return np.float32(lib().orc_tree_sum(_p(x)))


def variance(s, sq, n) -> np.float32:
    return np.float32(lib().orc_variance(float(s), float(sq), float(n)))


def top_k(var, n_hi: int) -> np.ndarray:
    var = _c(var, np.float32)
    out = np.zeros(128, np.uint8)
    lib().orc_top_k(_p(var), n_hi, _p(out))
    return out.astype(bool)


def key_pos(col: int, t: int, words_per_lane: int = 8):
    w, b = ctypes.c_int(), ctypes.c_int()
    lib().orc_key_pos(col, t, words_per_lane, ctypes.byref(w), ctypes.byref(b))
    return w.value, b.value


def key_pos4(col: int, t: int, words_per_lane: int = 16):
    """Word and bit of a 4-bit Key code (the (8, 4) configuration's planes)."""
    w, b = ctypes.c_int(), ctypes.c_int()
    lib().orc_key_pos4(col, t, words_per_lane, ctypes.byref(w), ctypes.byref(b))
    return w.value, b.value


def val_pos(t: int, c: int):
    w, b = ctypes.c_int(), ctypes.c_int()
    lib().orc_val_pos(t, c, ctypes.byref(w), ctypes.byref(b))
    return w.value, b.value


def val_pos4(t: int, c: int):
    """4-bit Value plane: (word, bit) of token t, channel c."""
    w, b = ctypes.c_int(), ctypes.c_int()
    lib().orc_val_pos4(t, c, ctypes.byref(w), ctypes.byref(b))
    return w.value, b.value


def quantize_page_f32(xk, xv, n_hi: int, running=None, lo_bit: int = 2, v_bit: int = 2):
    """One page-head from fp32 [32,128] tiles.  running = (sum[128], sumsq[128],
    count[1]) arrays updated in place, or None for page mode.  Returns
    (blob bytes, status)."""
    xk = _c(xk, np.float32)
    xv = _c(xv, np.float32)
    blob = np.zeros(page_bytes(n_hi, lo_bit, v_bit), np.uint8)
    if running is None:
        st = lib().orc_quantize_page_f32(_p(xk), _p(xv), n_hi, 0, None, None, None, _p(blob), lo_bit,
                                         v_bit)
    else:
        rs, rq, rc = running
        st = lib().orc_quantize_page_f32(_p(xk), _p(xv), n_hi, 1, _p(rs), _p(rq), _p(rc), _p(blob),
                                         lo_bit, v_bit)
    return blob, st


def page_channels(blob, n_hi: int, lo_bit: int = 2) -> np.ndarray:
    """The boosted channel list of a blob, row order (ascending ids)."""
    blob = _c(blob, np.uint8)
    out = np.zeros(max(n_hi, 1), np.int32)
    lib().orc_page_channels(_p(blob), n_hi, _p(out), lo_bit)
    return out[:n_hi]


def meta_pos(kind: str, a: int, b: int = 0) -> int:
    """Storage index of Key minima ("km", channel a), Value metadata ("vmeta",
    group a, token b) or channel-list rows ("kch", row a)."""
    pos = ctypes.c_int()
    lib().orc_meta_pos({"km": 0, "vmeta": 1, "kch": 2}[kind], a, b, ctypes.byref(pos))
    return pos.value


def dequant_page(blob, n_hi: int, lo_bit: int = 2, v_bit: int = 2):
    blob = _c(blob, np.uint8)
    kh = np.zeros((32, 128), np.float64)
    vh = np.zeros((32, 128), np.float64)
    st = ctypes.c_int()
    lib().orc_dequant_page(_p(blob), n_hi, _p(kh), _p(vh), ctypes.byref(st), lo_bit, v_bit)
    return kh, vh, st.value


def quantize_pages(Hkv, n_hi, rank_mode, in_dtype, k, v, page_ids, pool, pool_pages,
                   seq_of_page=None, n_seqs=0, run_sum=None, run_sumsq=None, run_count=None,
                   lo_bit=2, v_bit=2):
    """k, v: uint16 [n_pages*32, Hkv, 128]; pool: uint8 array updated in place."""
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    page_ids = _c(page_ids, np.int32)
    n_pages = page_ids.size
    sop = None if seq_of_page is None else _c(seq_of_page, np.int32)
    assert pool.flags.c_contiguous and pool.dtype == np.uint8
    return lib().orc_quantize_pages(Hkv, n_hi, rank_mode, in_dtype, _p(k), _p(v), n_pages,
                                    _p(page_ids), _p(sop), n_seqs, _p(run_sum), _p(run_sumsq),
                                    _p(run_count), _p(pool), pool_pages, lo_bit, v_bit)


def append_token(Hkv, n_hi, rank_mode, in_dtype, k_new, v_new, tail_k, tail_v, tail_len,
                 run_sum, run_sumsq, run_count, flush_page_ids, block_table, max_pages,
                 num_pages, pool, pool_pages, lo_bit=2, v_bit=2):
    """All state arrays are numpy arrays updated in place."""
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    fl = _c(flush_page_ids, np.int32)
    B = tail_len.size
    return lib().orc_append_token(Hkv, n_hi, rank_mode, in_dtype, _p(k_new), _p(v_new),
                                  _p(tail_k), _p(tail_v), _p(tail_len), _p(run_sum),
                                  _p(run_sumsq), _p(run_count), _p(fl), _p(block_table),
                                  max_pages, _p(num_pages), _p(pool), pool_pages, B, lo_bit,
                                  v_bit)


def decode_attention(Hkv, Hq, n_hi, in_dtype, q, pool, pool_pages, block_table, num_pages,
                     tail_k, tail_v, tail_len, sm_scale, lo_bit=2, v_bit=2):
    """Returns (out float64 [B, Hq, 128], status)."""
    q = _c(q, np.uint16)
    block_table = _c(block_table, np.int32)
    num_pages = _c(num_pages, np.int32)
    tail_len = _c(tail_len, np.int32)
    B = num_pages.size
    max_pages = block_table.shape[1] if block_table.ndim == 2 else 0
    tail_k = _c(tail_k, np.uint16)
    tail_v = _c(tail_v, np.uint16)
    out = np.zeros((B, Hq, 128), np.float64)
    st = lib().orc_decode_attention(Hkv, Hq, n_hi, in_dtype, _p(q), _p(pool), pool_pages,
                                    _p(block_table), max_pages, _p(num_pages), _p(tail_k),
                                    _p(tail_v), _p(tail_len), float(sm_scale), B, _p(out), lo_bit,
                                    v_bit)
    return out, st


def decode_f16kv(Hkv, Hq, in_dtype, q, pool, pool_pages, block_table, ctx_len, sm_scale):
    """16-bit paged KV baseline: pool uint16 [pool_pages, Hkv, 2, 32, 128] (K then V);
    returns (out float64 [B, Hq, 128], status)."""
    q = _c(q, np.uint16)
    pool = _c(pool, np.uint16)
    block_table = _c(block_table, np.int32)
    ctx_len = _c(ctx_len, np.int32)
    B = ctx_len.size
    max_pages = block_table.shape[1] if block_table.ndim == 2 else 0
    out = np.zeros((B, Hq, 128), np.float64)
    st = lib().orc_decode_f16kv(Hkv, Hq, in_dtype, _p(q), _p(pool), pool_pages, _p(block_table),
                                max_pages, _p(ctx_len), float(sm_scale), B, _p(out))
    return out, st


def decode_attention_one(Hkv, Hq, n_hi, in_dtype, q, pool, pool_pages, block_table, num_pages,
                         tail_k, tail_v, tail_len, sm_scale, b, kvh, lo_bit=2, v_bit=2):
    """The g = Hq/Hkv query heads of (sequence b, kv head kvh): (out [g, 128], status)."""
    g = Hq // Hkv
    out = np.zeros((g, 128), np.float64)
    max_pages = block_table.shape[1]
    st = lib().orc_decode_attention_one(Hkv, Hq, n_hi, in_dtype, _p(q), _p(pool), pool_pages,
                                        _p(block_table), max_pages, _p(num_pages), _p(tail_k),
                                        _p(tail_v), _p(tail_len), float(sm_scale), b, kvh, _p(out),
                                        lo_bit, v_bit)
    return out, st
