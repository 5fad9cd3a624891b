"""GPU parity on the quantizer's edge cases and the decode's error paths, through
the C ABI, against the CPU oracle.

* Ranking ties at the n_hi cut (equal variances; the lower channels win) in
  page, running and sequence statistics, for 2-bit and 4-bit Key planes
  (VeloxQuant-MLX docs, "How it works", Prefill step 2: the top
  hi_fraction * D channels).
* Values exactly halfway between two quantization levels at steps that are not
  powers of two, for 3, 15 and 255 levels (same page, Prefill step 3:
  asymmetric min/max groups): the kernel's approximate quotient must hand every
  such value to the correctly rounded division.
* A finite bf16 input beyond the fp16 range of the metadata, and a bf16 query
  beyond the fp16 range of the tensor-core operands: KITTY_ST_RANGE.
* A page wait bounded to one poll: KITTY_ST_TIMEOUT, the call returns, and the
  next call on the same context is exact.
"""

import dataclasses

import numpy as np
import pytest

import oracle
from mixed_precision_bit_gb300 import synth
from tests.edge_inputs import plant_half_way, plant_ties
from tests.kitty_cases import (attn_error, cfg_for, dev16, dev32, gpu_decode, gpu_quantize,
                               oracle_decode, oracle_quantize)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixed_precision_bit_gb300 import kitty
    kitty.load()


def _w(**kw):
    base = dataclasses.replace(synth.workload("small_gqa"), pages=np.array([3, 2, 4]),
                               tails=np.array([5, 0, 9]))
    return dataclasses.replace(base, **kw)


def _same_pool(w, inp, mode):
    pool, run = gpu_quantize(w, inp, mode=mode)
    ref, ref_run, st = oracle_quantize(w, inp, mode=mode)
    assert st == 0
    got = pool.cpu().numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, "first mismatching bytes at %s" % bad[:8]
    if run is not None:
        for g, r in zip(run, ref_run):
            assert (g.cpu().numpy().view(np.uint32) == r.view(np.uint32)).all()
    return pool, ref


@pytest.mark.parametrize("lo_bit", [2, 4])
@pytest.mark.parametrize("mode", [0, 1, 2], ids=["page", "running", "sequence"])
@pytest.mark.parametrize("roles", [(0, 40, 32), (20, 30, 32), (5, 20, 16)],
                         ids=["40tied-nhi32", "20+30tied-nhi32", "5+20tied-nhi16"])
def test_quantize_ties_bit_exact(roles, mode, lo_bit):
    """Equal variances straddling the n_hi cut: pools (codes, channel lists,
    steps, minima) and running totals bit-exact with the oracle, and the boosted
    lists are the larger-variance channels plus the lowest tied ones."""
    n_distinct, n_tied, n_hi = roles
    w = _w(n_hi=n_hi, lo_bit=lo_bit)
    inp = synth.host_inputs(w, seed=31)
    plant = plant_ties(inp, w, seed=32, n_distinct=n_distinct, n_tied=n_tied)
    _, ref = _same_pool(w, inp, mode)
    blob = oracle.page_bytes(n_hi, lo_bit)
    for i, pid in enumerate(inp["page_ids"]):
        b = int(inp["seq_of_page"][i])
        for h in range(w.Hkv):
            d, t = plant[(b, h)]
            o = (int(pid) * w.Hkv + h) * blob
            got = oracle.page_channels(ref[o:o + blob], n_hi, lo_bit)
            assert (got == np.sort(np.concatenate([d, t[:n_hi - n_distinct]]))).all()


@pytest.mark.parametrize("dtype", [synth.BF16, synth.F16], ids=["bf16", "f16"])
@pytest.mark.parametrize("lo_bit,n_hi,v_bit", [(2, 0, 2), (2, 32, 2), (2, 128, 2), (4, 0, 2),
                                               (4, 32, 2), (4, 128, 2), (4, 0, 4), (4, 32, 4)])
def test_quantize_rounding_ties_bit_exact(lo_bit, n_hi, v_bit, dtype):
    """Every Key channel and Value group holds values exactly halfway between two
    levels (3 and 15 levels at (4, 2); 15 and 255 at (8, 4); 3 or 15 for 2-bit or
    4-bit Values): bit-exact pools in page and running mode, then decode within
    tolerance."""
    levels = (3, 15) if lo_bit == 2 else (15, 255)
    w = _w(n_hi=n_hi, lo_bit=lo_bit, dtype=dtype, v_bit=v_bit)
    inp = synth.host_inputs(w, seed=33)
    boosted = np.sort(np.random.default_rng(34).permutation(128)[:n_hi])
    plant_half_way(inp, w, levels, boosted, seed=35, value_levels=(1 << v_bit) - 1)
    for mode in (0, 1):
        pool, ref = _same_pool(w, inp, mode)
        if mode == 0 and 0 < n_hi < 128:
            blob = oracle.page_bytes(n_hi, lo_bit, v_bit)
            assert (oracle.page_channels(ref[:blob], n_hi, lo_bit) == boosted).all()
    got = gpu_decode(w, inp, pool)
    want, _ = oracle_decode(w, inp, pool.cpu().numpy())
    assert attn_error(got, want)[0] <= 0


@pytest.mark.parametrize("mode", [0, 1], ids=["page", "running"])
def test_quantize_finite_bf16_beyond_fp16_range(mode):
    """A finite bf16 input above 65504 cannot be held by the fp16 step and
    minimum: KITTY_ST_RANGE (and the oracle agrees)."""
    import torch
    w = _w()
    inp = synth.host_inputs(w, seed=36)
    inp["k"][40, 1, 77] = synth.to_bits(np.array([70000.0]), synth.BF16)[0]
    inp["v"][3, 0, 5] = synth.to_bits(np.array([-1.0e5]), synth.BF16)[0]
    assert synth.from_bits(inp["k"][40, 1, 77:78], synth.BF16)[0] > 65504
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_quantize(w, inp, mode=mode, status=st)
    _, _, ost = oracle_quantize(w, inp, mode=mode)
    assert int(st.item()) == oracle.ST["RANGE"] == ost


@pytest.mark.parametrize("bad,code", [(70000.0, "RANGE"), (float("nan"), "NONFINITE"),
                                      (float("-inf"), "NONFINITE")])
@pytest.mark.parametrize("Hq", [8, 16], ids=["g4", "g8"])
def test_decode_query_beyond_fp16_range(bad, code, Hq):
    """The tensor cores take the query as fp16: a bf16 query element above 65504
    (or non-finite) is reported; an in-range query of the same batch reports
    nothing."""
    import torch
    w = _w(Hq=Hq)
    inp = synth.host_inputs(w, seed=37)
    pool, _ = gpu_quantize(w, inp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_decode(w, inp, pool, status=st)
    assert int(st.item()) == 0
    inp["q"][2, 5, 100] = synth.to_bits(np.array([bad]), synth.BF16)[0]
    gpu_decode(w, inp, pool, status=st)
    assert int(st.item()) == oracle.ST[code]


@pytest.mark.parametrize("Hq", [32, 64], ids=["g4", "g8"])
def test_decode_wait_timeout_reports_and_returns(Hq):
    """A page wait bounded to one poll of its barrier runs out on ordinary copies
    (the pool is evicted from L2 first): KITTY_ST_TIMEOUT is reported, the call
    completes (the CTA drains its copies in flight before it exits), and the
    next call with the library's bound on the same context gives the same bytes
    as a call before the timeout."""
    import torch
    from mixed_precision_bit_gb300 import kitty
    w = dataclasses.replace(synth.workload("small_gqa"), B=16, Hq=Hq, Hkv=8,
                            pages=np.full(16, 48), tails=np.full(16, 3))
    inp = synth.host_inputs(w, seed=38)
    pool, _ = gpu_quantize(w, inp)
    before = gpu_decode(w, inp, pool)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")   # > 3x L2
    cfg = cfg_for(w)
    cfg.decode_wait_polls = 1
    bt = inp["block_table"]
    ws = torch.empty(max(kitty.decode_workspace_bytes(cfg, w.B, bt.shape[1]), 16) // 4,
                     dtype=torch.float32, device="cuda")
    out = torch.empty((w.B, w.Hq, 128), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    flush.fill_(1)
    kitty.decode_attention(cfg, dev16(inp["q"]), pool, inp["pool_pages"], dev32(bt),
                           dev32(inp["num_pages"]), dev16(inp["tail_k"]), dev16(inp["tail_v"]),
                           dev32(inp["tail_len"]), float(np.float32(1 / np.sqrt(128))), out,
                           workspace=ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == kitty.ST["TIMEOUT"]
    st.zero_()
    after = gpu_decode(w, inp, pool, status=st)
    assert int(st.item()) == 0
    assert np.array_equal(before, after)
    ref, _ = oracle_decode(w, inp, pool.cpu().numpy())
    assert attn_error(after, ref)[0] <= 0
