"""The C ABI library builds, loads and exports every declared entry point; its
host-only parts (sizes, effective bits, page allocator, argument checks) work
without a GPU."""

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def K():
    from mixed_precision_bit_gb300 import kitty
    kitty.load()
    return kitty


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^(?:int|int32_t|float|void)\s+\*?(kitty_[a-z_0-9]+)\s*\(",
                                    src, re.M))
    return names


def test_exports_every_declared_symbol(K):
    names = _declared()
    assert {"kitty_quantize_pages", "kitty_append_token", "kitty_decode_attention"} <= names
    lib = K.load()
    for n in names:
        assert hasattr(lib, n), n
    assert set(K.EXPORTS) == names
    assert lib.kitty_abi_version() == 5


def test_page_bytes_and_avg_bits(K):
    for n_hi, blob in ((32, 3360), (16, 3216), (0, 3072), (128, 4224)):
        cfg = K.Config(num_kv_heads=8, num_q_heads=32, n_hi=n_hi)
        assert K.page_bytes(cfg) == (blob, 8 * blob)
    assert K.avg_bits(K.Config(8, 32, n_hi=32)) == 2.5
    assert K.avg_bits(K.Config(8, 32, n_hi=0)) == 2.0
    assert K.avg_bits(K.Config(8, 32, n_hi=64)) == 3.0
    # (hi_bit, lo_bit) = (8, 4): two 4-bit Key planes; the table's (0.25, 8, 4) row is 5.0 bits
    import oracle
    for n_hi in (0, 16, 32, 128):
        cfg = K.Config(num_kv_heads=8, num_q_heads=32, n_hi=n_hi, hi_bit=8, lo_bit=4)
        blob = oracle.page_bytes(n_hi, 4)
        assert K.page_bytes(cfg) == (blob, 8 * blob)
    assert K.avg_bits(K.Config(8, 32, n_hi=32, hi_bit=8, lo_bit=4)) == 5.0


def test_config_checks(K):
    for bad, code in ((dict(n_hi=8), -2), (dict(head_dim=64), -2), (dict(hi_bit=8), -2),
                      (dict(lo_bit=4), -2), (dict(hi_bit=6, lo_bit=3), -2),
                      (dict(num_q_heads=12), -1), (dict(in_dtype=7), -1),
                      (dict(v_bit=4), -2), (dict(v_bit=3, hi_bit=8, lo_bit=4), -2)):
        cfg = K.Config(**{**dict(num_kv_heads=8, num_q_heads=32), **bad})
        with pytest.raises(K.KittyError) as e:
            K.page_bytes(cfg)
        assert e.value.code == code
    # query groups: decode takes g <= 32 (head groups of 4), the fused append + decode g <= 4
    cfg = K.Config(num_kv_heads=8, num_q_heads=64)   # g = 8
    K.page_bytes(cfg)
    assert K.decode_workspace_bytes(cfg, 4, 16) >= 0
    lib = K.load()
    rc = lib.kitty_append_decode(ctypes.byref(cfg.c()), *([None] * 11), 16, None, None, 1, 0.1,
                                 None, 0, None, 0, 1, None, None)
    assert rc == -2
    cfg = K.Config(num_kv_heads=1, num_q_heads=33)   # g = 33: quantize ok, decode unsupported
    K.page_bytes(cfg)
    with pytest.raises(K.KittyError):
        K.decode_workspace_bytes(cfg, 4, 16)
    # 4-bit Values with 4-bit Key planes: the Value plane doubles
    cfg = K.Config(num_kv_heads=8, num_q_heads=32, n_hi=0, hi_bit=8, lo_bit=4, v_bit=4)
    assert K.page_bytes(cfg) == (5120, 8 * 5120)


def test_allocator(K):
    a = K.PageAllocator(6)
    assert list(a.alloc(3)) == [0, 1, 2] and a.free_count == 3
    with pytest.raises(K.KittyError) as e:
        a.alloc(4)
    assert e.value.code == -5 and a.free_count == 3
    a.free([1])
    assert list(a.alloc(1)) == [1]
    with pytest.raises(K.KittyError):
        a.free([5])          # not allocated
    with pytest.raises(K.KittyError):
        a.free([0, 0])       # duplicate
    assert a.free_count == 3
    a.free([0, 1, 2])
    assert a.free_count == 6
    a.close()


def test_null_arguments_rejected_before_launch(K):
    """Argument errors come back synchronously and nothing is launched."""
    lib = K.load()
    cfg = K.Config(num_kv_heads=1, num_q_heads=1).c()
    rc = lib.kitty_quantize_pages(ctypes.byref(cfg), None, None, 1, None, None, 0, None, None,
                                  None, None, 1, None, None)
    assert rc == -1
    rc = lib.kitty_decode_attention(ctypes.byref(cfg), None, None, 1, None, 1, None, None, None,
                                    None, 0.1, None, 0, None, 0, 1, None, None)
    assert rc == -1
    assert lib.kitty_quantize_pages(ctypes.byref(cfg), None, None, 0, None, None, 0, None, None,
                                    None, None, 0, None, None) == 0   # empty batch: no-op


def test_decode_plan_and_workspace(K):
    cfg = K.Config(num_kv_heads=8, num_q_heads=32)
    s, c = K.decode_plan(cfg, 16, 128)
    assert 1 <= s <= 256 and s * c >= 128 and c % 8 == 0 and c >= 16
    assert K.decode_workspace_bytes(cfg, 16, 128) == (16 * 32 * s * 132 * 4 if s > 1 else 0)
    for B, M in ((1, 4096), (177, 256), (4096, 256), (1, 3), (64, 65536)):
        s, c = K.decode_plan(cfg, B, M)
        assert 1 <= s <= 256 and c <= M and s * c >= M, (B, M, s, c)
    assert K.decode_plan(cfg, 5, 0)[0] == 1
    # planning hint: the batch's total pages; pieces stay within one slot's fair share
    for B, M, tot in ((8, 2048, 8 * 1280), (64, 256, 64 * 256), (177, 257, 177 * 256)):
        h = K.Config(num_kv_heads=8, num_q_heads=32, decode_total_pages=tot)
        s, c = K.decode_plan(h, B, M)
        assert 1 <= s <= 256 and c <= M and s * c >= M, (B, M, s, c)
    with pytest.raises(K.KittyError):
        K.decode_plan(K.Config(num_kv_heads=8, num_q_heads=32, decode_total_pages=-1), 4, 16)
    # planning hint: the longest sequence; the splits still cover the whole table
    for B, M, mx in ((16, 136, 128), (64, 264, 256), (8, 2048, 2000), (4, 100, 1000), (3, 50, 1)):
        h = K.Config(num_kv_heads=8, num_q_heads=32, decode_total_pages=B * min(M, mx),
                     decode_max_pages=mx)
        s, c = K.decode_plan(h, B, M)
        assert 1 <= s <= 256 and c <= M, (B, M, mx, s, c)
        assert K.decode_workspace_bytes(h, B, M) == (B * 32 * s * 132 * 4 if s > 1 else 0)
    # a 16 x 128-page batch in a 136-page table: four 32-page splits, the last to the end
    h = K.Config(num_kv_heads=8, num_q_heads=32, decode_total_pages=16 * 128, decode_max_pages=128)
    assert K.decode_plan(h, 16, 136) == (4, 40)
    # equal lengths and few units: one wave of equal splits (without a device the
    # planner counts 148 SMs: 4 resident CTAs each, 3 for 8 query heads per CTA)
    h = K.Config(num_kv_heads=8, num_q_heads=64, decode_total_pages=16 * 256, decode_max_pages=256)
    assert K.decode_plan(h, 16, 257) == (3, 86)      # 128 units of 8 heads, 444 slots: 86, 86, 84 + 1
    h = K.Config(num_kv_heads=8, num_q_heads=32, decode_total_pages=8 * 256, decode_max_pages=256)
    assert K.decode_plan(h, 8, 256) == (9, 29)       # 64 units, 592 slots: nine splits of 29 or fewer
    # the same total with unequal lengths keeps the longest-first sizes (largest first)
    h = K.Config(num_kv_heads=8, num_q_heads=32, decode_total_pages=8 * 256 - 1, decode_max_pages=256)
    s, c = K.decode_plan(h, 8, 256)
    assert (s, c) != (9, 29) and s * c >= 256
    with pytest.raises(K.KittyError):
        K.decode_plan(K.Config(num_kv_heads=8, num_q_heads=32, decode_max_pages=-1), 4, 16)
    cfg.decode_pages_per_split = 1000
    assert K.decode_plan(cfg, 16, 128) == (1, 128)
    assert K.decode_workspace_bytes(cfg, 16, 128) == 0
    cfg.decode_pages_per_split = 4
    assert K.decode_plan(cfg, 16, 128) == (32, 4)
    assert K.decode_plan(cfg, 16, 4096) == (256, 16)


def test_binding_refuses_host_and_strided_tensors():
    """The ctypes binding passes raw device addresses: a host tensor or a view
    with gaps is refused before any call."""
    import torch
    from mixed_precision_bit_gb300 import kitty as K
    with pytest.raises(ValueError, match="device memory"):
        K._ptr(torch.zeros(4, 4))
    assert K._ptr(None) is None
    assert K._ptr(1024).value == 1024


@pytest.mark.gpu
def test_binding_refuses_strided_device_tensor():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixed_precision_bit_gb300 import kitty as K
    with pytest.raises(ValueError, match="contiguous"):
        K._ptr(torch.zeros(4, 4, device="cuda").t())
