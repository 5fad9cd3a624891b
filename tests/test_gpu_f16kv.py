"""GPU parity of the 16-bit paged KV baseline (the unquantized layout of the
paper's same-budget comparison, Abstract) against the fp64 oracle, through the
C ABI: page writes and appends bit-exact, decode attention within 2e-3 * RMS
(+ half an output ulp for 16-bit outputs)."""

import numpy as np
import pytest

import oracle
from mixed_precision_bit_gb300 import synth
from tests.kitty_cases import attn_error, dev16, dev32

pytestmark = pytest.mark.gpu
P, D = 32, 128


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixed_precision_bit_gb300 import kitty
    kitty.load()


def _cfg(Hkv, Hq, dt):
    from mixed_precision_bit_gb300 import kitty
    return kitty.Config(num_kv_heads=Hkv, num_q_heads=Hq, in_dtype=dt)


def _cache(Hkv, Hq, dt, lens, seed, spare=0):
    """Host pool, block table and per-sequence tokens; pages written on the GPU."""
    import torch
    from mixed_precision_bit_gb300 import kitty
    r = np.random.default_rng(seed)
    B = len(lens)
    npg = [(int(L) + P - 1) // P for L in lens]
    max_pages = max(max(npg), 1) + spare
    pool_pages = sum(npg) + B * spare + 1
    ids = r.permutation(pool_pages).astype(np.int32)
    bt = np.full((B, max_pages), -1, np.int32)
    k = synth.to_bits(r.standard_normal((max(sum(npg), 1) * P, Hkv, D)) * np.exp(r.standard_normal(D)), dt)
    v = synth.to_bits(r.standard_normal((max(sum(npg), 1) * P, Hkv, D)), dt)
    page_ids = np.zeros(sum(npg), np.int32)
    off = 0
    for b in range(B):
        bt[b, :npg[b]] = ids[off:off + npg[b]]
        page_ids[off:off + npg[b]] = ids[off:off + npg[b]]
        off += npg[b]
    cfg = _cfg(Hkv, Hq, dt)
    _, per_page = kitty.f16kv_page_bytes(cfg)
    pool = torch.zeros(pool_pages * per_page, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if page_ids.size:
        kitty.f16kv_write_pages(cfg, dev16(k), dev16(v), dev32(page_ids), pool, pool_pages, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # host mirror of the pool
    host = np.zeros((pool_pages, Hkv, 2, P, D), np.uint16)
    for i, pid in enumerate(page_ids):
        host[pid, :, 0] = k[i * P:(i + 1) * P].transpose(1, 0, 2)
        host[pid, :, 1] = v[i * P:(i + 1) * P].transpose(1, 0, 2)
    got = pool.cpu().numpy().view(np.uint16).reshape(host.shape)
    assert (got == host).all(), "written pages differ"
    q = synth.to_bits(r.standard_normal((B, Hq, D)), dt)
    return dict(cfg=cfg, pool=pool, host=host, bt=bt, lens=np.asarray(lens, np.int32), q=q,
                pool_pages=pool_pages, ids=ids, used=off)


def _decode(c, out_dtype="f32", status=None):
    import torch
    from mixed_precision_bit_gb300 import kitty
    dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[out_dtype]
    B, Hq = c["q"].shape[:2]
    out = torch.full((B, Hq, D), float("nan"), dtype=dt, device="cuda")
    n = kitty.f16kv_workspace_bytes(c["cfg"], B, c["bt"].shape[1])
    ws = torch.empty(max(n, 16) // 4, dtype=torch.float32, device="cuda")
    kitty.f16kv_decode(c["cfg"], dev16(c["q"]), c["pool"], c["pool_pages"], dev32(c["bt"]),
                       dev32(c["lens"]), float(np.float32(1 / np.sqrt(D))), out, workspace=ws,
                       status=status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def _oracle(c):
    Hkv = c["cfg"].num_kv_heads
    return oracle.decode_f16kv(Hkv, c["cfg"].num_q_heads, c["cfg"].in_dtype, c["q"], c["host"],
                               c["pool_pages"], c["bt"], c["lens"], float(np.float32(1 / np.sqrt(D))))


CASES = [
    (2, 8, synth.BF16, [70, 1, 0, 64, 33]),       # partial pages, a single token, empty
    (2, 8, synth.F16, [70, 1, 0, 64, 33]),
    (2, 2, synth.BF16, [200, 31, 32]),            # g = 1
    (3, 6, synth.BF16, [95, 128]),                # g = 2
    (1, 3, synth.F16, [257]),                     # g = 3
    (4, 16, synth.BF16, [1000, 2047, 5]),         # several splits
]


@pytest.mark.parametrize("case", CASES, ids=["c%d" % i for i in range(len(CASES))])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16", "f16"])
def test_f16kv_decode_matches_oracle(case, out_dtype):
    import torch
    Hkv, Hq, dt, lens = case
    c = _cache(Hkv, Hq, dt, lens, seed=41)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _decode(c, out_dtype, status=st)
    ref, ost = _oracle(c)
    assert int(st.item()) == ost
    excess, rel = attn_error(got, ref, out_dtype)
    assert excess <= 0, "max err %.3e of RMS" % rel
    for b, L in enumerate(lens):
        if L == 0:
            assert (got[b] == 0).all()


def test_f16kv_append_matches_host_model():
    """Tokens appended one at a time, starting new pages at the caller's ids:
    pool, block table and lengths bit-exact with a host model, then decode
    within tolerance of the oracle."""
    import torch
    from mixed_precision_bit_gb300 import kitty
    Hkv, Hq, dt = 2, 8, synth.BF16
    lens = [30, 0, 64, 5]
    c = _cache(Hkv, Hq, dt, lens, seed=42, spare=3)
    B = len(lens)
    r = np.random.default_rng(43)
    free = [int(x) for x in c["ids"][c["used"]:]]
    bt_d, len_d = dev32(c["bt"]), dev32(c["lens"])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    host, bt, ln = c["host"], c["bt"], c["lens"].copy()
    for step in range(40):
        kn = synth.to_bits(r.standard_normal((B, Hkv, D)), dt)
        vn = synth.to_bits(r.standard_normal((B, Hkv, D)), dt)
        new = np.full(B, -1, np.int32)
        for b in range(B):
            if ln[b] % P == 0:
                new[b] = free.pop()
        kitty.f16kv_append(c["cfg"], dev16(kn), dev16(vn), c["pool"], c["pool_pages"], bt_d, len_d,
                           dev32(new), status=st)
        for b in range(B):
            if ln[b] % P == 0:
                bt[b, ln[b] // P] = new[b]
            pid = bt[b, ln[b] // P]
            host[pid, :, 0, ln[b] % P] = kn[b]
            host[pid, :, 1, ln[b] % P] = vn[b]
            ln[b] += 1
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert (bt_d.cpu().numpy() == bt).all() and (len_d.cpu().numpy() == ln).all()
    got_pool = c["pool"].cpu().numpy().view(np.uint16).reshape(host.shape)
    for b in range(B):
        for p in bt[b][bt[b] >= 0]:
            assert (got_pool[p] == host[p]).all(), (b, p)
    c["lens"] = ln
    got = _decode(c)
    ref, _ = _oracle(c)
    assert attn_error(got, ref)[0] <= 0


def test_f16kv_bad_page_sets_status():
    import torch
    c = _cache(2, 8, synth.BF16, [70, 64], seed=44)
    c["bt"] = c["bt"].copy()
    c["bt"][0, 1] = c["pool_pages"] + 5
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _decode(c, status=st)
    assert int(st.item()) == oracle.ST["BAD_PAGE"]
