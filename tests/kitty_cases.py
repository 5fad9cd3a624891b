"""Shared helpers for the GPU parity tests: run a workload through the library
(C ABI via the ctypes binding) and through the oracle on the same host inputs."""

from __future__ import annotations

import math

import numpy as np

import oracle
from mixed_precision_bit_gb300 import synth

TOL_REL = 2e-3   # max |gpu - oracle| <= 2e-3 * RMS(oracle output)


def cfg_for(w, rank_mode=0, pps=0):
    from mixed_precision_bit_gb300 import kitty
    return kitty.Config(num_kv_heads=w.Hkv, num_q_heads=w.Hq, n_hi=w.n_hi, in_dtype=w.dtype,
                        rank_mode=rank_mode, decode_pages_per_split=pps,
                        hi_bit=2 * w.lo_bit, lo_bit=w.lo_bit, v_bit=w.v_bit)


def dev16(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def dev32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def gpu_quantize(w, inp, running=False, status=None, mode=None):
    """Quantize every page on the GPU; returns (pool uint8 tensor, run state or None).
    mode: 0 page, 1 running, 2 sequence (default: running if `running` else page)."""
    import torch
    from mixed_precision_bit_gb300 import kitty
    mode = (1 if running else 0) if mode is None else mode
    running = mode != 0
    cfg = cfg_for(w, rank_mode=mode)
    blob, per_page = kitty.page_bytes(cfg)
    pool = torch.zeros(inp["pool_pages"] * per_page, dtype=torch.uint8, device="cuda")
    run = None
    args = {}
    if running:
        run = (torch.zeros((w.B, w.Hkv, 128), dtype=torch.float32, device="cuda"),
               torch.zeros((w.B, w.Hkv, 128), dtype=torch.float32, device="cuda"),
               torch.zeros((w.B, w.Hkv), dtype=torch.int32, device="cuda"))
        args = dict(seq_of_page=dev32(inp["seq_of_page"]), n_seqs=w.B, run_sum=run[0],
                    run_sumsq=run[1], run_count=run[2])
    if inp["page_ids"].size:
        kitty.quantize_pages(cfg, dev16(inp["k"]), dev16(inp["v"]), dev32(inp["page_ids"]), pool,
                             inp["pool_pages"], status=status, **args)
    torch.cuda.synchronize()
    return pool, run


def oracle_quantize(w, inp, running=False, mode=None):
    mode = (1 if running else 0) if mode is None else mode
    running = mode != 0
    pool = np.zeros(inp["pool_pages"] * w.Hkv * oracle.page_bytes(w.n_hi, w.lo_bit, w.v_bit), np.uint8)
    if running:
        rs = np.zeros((w.B, w.Hkv, 128), np.float32)
        rq = np.zeros_like(rs)
        rc = np.zeros((w.B, w.Hkv), np.int32)
        st = oracle.quantize_pages(w.Hkv, w.n_hi, mode, w.dtype, inp["k"], inp["v"], inp["page_ids"],
                                   pool, inp["pool_pages"], seq_of_page=inp["seq_of_page"],
                                   n_seqs=w.B, run_sum=rs, run_sumsq=rq, run_count=rc,
                                   lo_bit=w.lo_bit, v_bit=w.v_bit)
        return pool, (rs, rq, rc), st
    st = oracle.quantize_pages(w.Hkv, w.n_hi, 0, w.dtype, inp["k"], inp["v"], inp["page_ids"],
                               pool, inp["pool_pages"], lo_bit=w.lo_bit, v_bit=w.v_bit)
    return pool, None, st


def gpu_decode(w, inp, pool, out_dtype="f32", pps=0, status=None, sm_scale=None, out_offset=0):
    """out_offset: the output array starts that many elements into its buffer."""
    import torch
    from mixed_precision_bit_gb300 import kitty
    cfg = cfg_for(w, pps=pps)
    dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[out_dtype]
    n = w.B * w.Hq * 128
    out = torch.full((n + out_offset,), float("nan"), dtype=dt, device="cuda")[out_offset:]
    out = out.view(w.B, w.Hq, 128)
    bt = inp["block_table"]
    nbytes = kitty.decode_workspace_bytes(cfg, w.B, bt.shape[1])
    ws = torch.empty(max(nbytes, 16) // 4, dtype=torch.float32, device="cuda")
    sm = float(np.float32(1 / math.sqrt(128))) if sm_scale is None else sm_scale
    kitty.decode_attention(cfg, dev16(inp["q"]), pool, inp["pool_pages"], dev32(bt),
                           dev32(inp["num_pages"]), dev16(inp["tail_k"]), dev16(inp["tail_v"]),
                           dev32(inp["tail_len"]), sm, out, workspace=ws, status=status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def oracle_decode(w, inp, pool, sm_scale=None):
    sm = float(np.float32(1 / math.sqrt(128))) if sm_scale is None else sm_scale
    return oracle.decode_attention(w.Hkv, w.Hq, w.n_hi, w.dtype, inp["q"], pool,
                                   inp["pool_pages"], inp["block_table"], inp["num_pages"],
                                   inp["tail_k"], inp["tail_v"], inp["tail_len"], sm,
                                   lo_bit=w.lo_bit, v_bit=w.v_bit)


def half_ulp(ref, out_dtype):
    if out_dtype == "f32":
        return 0.0
    mant = 7 if out_dtype == "bf16" else 10
    a = np.maximum(np.abs(ref), 2.0 ** -126)
    return 0.5 * 2.0 ** (np.floor(np.log2(a)) - mant)


def attn_error(got, ref, out_dtype="f32"):
    """(max excess over the bound, max |err| / RMS): passes when the first is <= 0."""
    rms = math.sqrt(float(np.mean(ref ** 2))) if ref.size else 0.0
    err = np.abs(got - ref)
    bound = TOL_REL * rms + half_ulp(ref, out_dtype)
    return float((err - bound).max()), float(err.max() / rms) if rms > 0 else float(err.max())
