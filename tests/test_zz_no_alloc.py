"""The allocation-free decode entry point, for callers that cannot allocate
device memory while they run (e.g. a server that reserved all GPU memory for its
page pool up front).  It must produce what kitty_decode_attention produces with
a caller workspace, call after call, although it keeps its split-K partials in
one fixed device array shared by every call.  This file sorts last so that a
run stopping at the first failure has run every other test first."""

import ctypes
import dataclasses

import numpy as np
import pytest

from mixed_precision_bit_gb300 import synth
from tests.kitty_cases import cfg_for, dev16, dev32, gpu_quantize

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run(kitty, cfg, w, inp, pool, noalloc, out_dtype):
    import torch
    dt = {"f32": torch.float32, "bf16": torch.bfloat16}[out_dtype]
    out = torch.full((w.B, w.Hq, 128), float("nan"), dtype=dt, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (cfg, dev16(inp["q"]), pool, inp["pool_pages"], dev32(inp["block_table"]),
            dev32(inp["num_pages"]), dev16(inp["tail_k"]), dev16(inp["tail_v"]),
            dev32(inp["tail_len"]), 0.08838834764831845, out)
    if noalloc:
        kitty.decode_attention_noalloc(*args, status=st)
    else:
        nbytes = kitty.decode_workspace_bytes(cfg, w.B, inp["block_table"].shape[1])
        ws = torch.empty(max(nbytes, 16) // 4, dtype=torch.float32, device="cuda")
        kitty.decode_attention(*args, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_noalloc_matches_workspace_entry_point(out_dtype):
    """Both entry points run the same kernels on the same split plan, so their
    outputs are the same bytes.  Calls with 16 splits and with the planner's few
    splits alternate on the one scratch array: partials a call leaves behind
    never reach a later call."""
    from mixed_precision_bit_gb300 import kitty
    kitty.load()
    w = dataclasses.replace(synth.workload("small_gqa"), pages=np.array([37, 1, 64]),
                            tails=np.array([0, 5, 17]))
    inp = synth.host_inputs(w, seed=11)
    pool, _ = gpu_quantize(w, inp)
    many, few = cfg_for(w, pps=4), cfg_for(w, pps=0)     # 16 splits; the planner's
    assert kitty.decode_plan(many, w.B, 64)[0] == 16
    assert 1 < kitty.decode_plan(few, w.B, 64)[0] < 16
    ref_many = _run(kitty, many, w, inp, pool, False, out_dtype)
    ref_few = _run(kitty, few, w, inp, pool, False, out_dtype)
    for cfg, ref in ((many, ref_many), (few, ref_few), (many, ref_many), (few, ref_few)):
        got = _run(kitty, cfg, w, inp, pool, True, out_dtype)
        assert np.array_equal(got, ref), "no-alloc output differs from the workspace path"

    t = synth.workload("tiny")                           # one split: no scratch used
    tin = synth.host_inputs(t, seed=11)
    tpool, _ = gpu_quantize(t, tin)
    ref = _run(kitty, cfg_for(t), t, tin, tpool, False, out_dtype)
    for _ in range(2):
        assert np.array_equal(_run(kitty, cfg_for(t), t, tin, tpool, True, out_dtype), ref)


def test_noalloc_rejects_batches_beyond_its_scratch():
    from mixed_precision_bit_gb300 import kitty
    lib = kitty.load()
    # 64 sequences x 32 heads x 256 splits of 132 floats is far beyond 8 MiB
    cfg = kitty.Config(num_kv_heads=8, num_q_heads=32, decode_pages_per_split=4)
    need = kitty.decode_workspace_bytes(cfg, 64, 1024)
    assert need > kitty.NOALLOC_SCRATCH_BYTES
    dummy = ctypes.c_void_p(16)   # never dereferenced: the call must refuse first
    rc = lib.kitty_decode_attention_noalloc(ctypes.byref(cfg.c()), dummy, dummy, 1, dummy, 1024,
                                            dummy, None, None, None, 0.1, dummy, 0, 64, None, None)
    assert rc == -4
