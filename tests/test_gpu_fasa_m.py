"""FASA-M placement (GPU): the K/V caches in page-locked host memory, the
dominant key cache in device memory ("Hardware-Aware Variants" on the FASA
pages).  The step reads the caches only in the row gather, so the results
must equal the all-device run bit for bit; the append step must also land
its row in host memory."""

import types

import numpy as np
import pytest

import oracle as O
from tests import parity as P
from tests.gpu_util import build_kdom, ensure_built, oracle_unit
from workload import configs, gpu_gen

pytestmark = pytest.mark.gpu


def _check_units(L, cfg, out, idx, cnt, units=None, budget=None):
    """Each (batch, KV head) unit of a step's results against the oracle on
    the stored inputs of layer-like L: the selected set (near-tie rule) and
    the output over that set."""
    k = cfg.budget if budget is None else budget
    G = cfg.group
    out, idx, cnt = (np.asarray(t.cpu().numpy() if hasattr(t, "cpu") else t) for t in (out, idx, cnt))
    if units is None:
        units = [(b, h) for b in range(cfg.batch) for h in range(cfg.n_kv_heads)]
    for b, h in units:
        ref = oracle_unit(L, b, h, k)
        n = int(L.seq_lens_host[b])
        assert cnt[b, h] == min(k, n)
        mine = idx[b, h, :cnt[b, h]]
        P.check_selection(mine, ref["scores"], k)
        fac = O.focused_attention_unit(ref["q_rot"], ref["K"], ref["V"], mine)
        P.check_output(out[b, h * G:(h + 1) * G], fac, cfg.dtype)


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    ensure_built()


def _ws(dims, budget):
    import torch
    from kv_cache_token_tip_gb300 import fasa_workspace_size
    n = fasa_workspace_size(dims, budget)
    return torch.empty(max(n, 16), dtype=torch.uint8, device="cuda") if n else None


@pytest.mark.parametrize("name,over", [("llama3_8b_ctx32k", dict(context=8192, batch=2)),
                                       ("qwen25_7b_b8_ctx16k", dict(context=4096, batch=2))])
def test_step_and_dense_with_host_caches(name, over):
    import torch
    from kv_cache_token_tip_gb300 import (dims_for, fasa_apply_rope_q, fasa_decode_step, fasa_dense_attention,
                                          fasa_device_status)
    cfg = configs.CONFIGS[name].with_(**over)
    L = gpu_gen.make_layer(cfg, 0)
    dims = dims_for(cfg)
    kd = build_kdom(L, dims)
    ws = _ws(dims, cfg.budget)
    Kh, Vh = L.k.cpu().pin_memory(), L.v.cpu().pin_memory()
    res = []
    for K, V in ((L.k, L.v), (Kh, Vh)):
        out = torch.full((cfg.batch, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=torch.float32, device="cuda")
        idx = torch.empty((cfg.batch, cfg.n_kv_heads, cfg.budget), dtype=torch.int32, device="cuda")
        cnt = torch.empty((cfg.batch, cfg.n_kv_heads), dtype=torch.int32, device="cuda")
        fasa_decode_step(L.q, L.pos, K, V, kd, L.dom_fc, L.seq_lens, cfg.budget, out, idx, cnt, ws, dims)
        q_rot = torch.empty_like(out)
        fasa_apply_rope_q(L.q, L.pos, q_rot, dims)
        dense = torch.empty_like(out)
        fasa_dense_attention(q_rot, K, V, L.seq_lens, dense, dims)
        assert fasa_device_status() == 0
        res.append((out.cpu(), idx.cpu(), dense.cpu(), cnt.cpu()))
    # the host-placement run against the oracle, unit by unit
    _check_units(L, cfg, res[1][0], res[1][1], res[1][3])
    G = cfg.group
    for b, h in ((0, 0), (cfg.batch - 1, cfg.n_kv_heads - 1)):
        ref = oracle_unit(L, b, h, cfg.budget)
        full = O.focused_attention_unit(ref["q_rot"], ref["K"], ref["V"], np.arange(int(L.seq_lens_host[b])))
        P.check_output(res[1][2].numpy()[b, h * G:(h + 1) * G], full, cfg.dtype)
    # and bit for bit the device-placement run
    assert torch.equal(res[0][1], res[1][1])
    assert torch.equal(res[0][0], res[1][0])
    assert torch.equal(res[0][2], res[1][2])


def test_append_step_with_host_caches():
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_decode_step_append, fasa_device_status
    cfg = configs.CONFIGS["llama3_8b_ctx32k"].with_(context=4096, batch=2)
    L = gpu_gen.make_layer(cfg, 0)
    L.seq_lens = torch.tensor([3000, 77], dtype=torch.int32, device="cuda")
    dims = dims_for(cfg)
    kd_dev = build_kdom(L, dims)
    kd_host_run = kd_dev.clone()
    gen = torch.Generator(device="cuda").manual_seed(9)
    shape = (cfg.batch, cfg.n_kv_heads, cfg.head_dim)
    kn = torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
    vn = torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
    ws = _ws(dims, cfg.budget)
    Kd, Vd = L.k.clone(), L.v.clone()
    Kh, Vh = L.k.cpu().pin_memory(), L.v.cpu().pin_memory()
    outs = []
    for K, V, kd in ((Kd, Vd, kd_dev), (Kh, Vh, kd_host_run)):
        out = torch.full((cfg.batch, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=torch.float32, device="cuda")
        idx = torch.empty((cfg.batch, cfg.n_kv_heads, cfg.budget), dtype=torch.int32, device="cuda")
        cnt = torch.empty((cfg.batch, cfg.n_kv_heads), dtype=torch.int32, device="cuda")
        fasa_decode_step_append(L.q, kn, vn, L.seq_lens, K, V, kd, L.dom_fc, cfg.budget, out, idx, cnt, ws, dims)
        assert fasa_device_status() == 0
        outs.append((out.cpu(), idx.cpu(), cnt.cpu()))
    # the host run against the oracle over the appended caches: len + 1
    # tokens, the query at position len
    lens = L.seq_lens.cpu().numpy()
    Lh = types.SimpleNamespace(cfg=cfg, q=L.q, k=Kh, v=Vh, seq_lens_host=lens + 1, pos_host=lens,
                               dom_fc_host=L.dom_fc_host)
    _check_units(Lh, cfg, *outs[1])
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(kd_dev, kd_host_run)
    assert torch.equal(Kd.cpu(), Kh) and torch.equal(Vd.cpu(), Vh)


def test_fasa_m_hbm_footprint_within_eq10():
    """With the caches in host memory, what the step keeps in HBM (K_dom, q,
    lengths, positions, the FC table, the output, the workspace) is within
    Eq. 10's estimate for the layer, and the library allocates no device
    memory of its own across steps."""
    import torch
    import oracle as O
    from kv_cache_token_tip_gb300 import dims_for, fasa_decode_step, fasa_device_status
    for name, over in (("llama3_8b_ctx32k", dict()), ("llama3_8b_b4_ctx128k", dict(batch=2))):
        cfg = configs.CONFIGS[name].with_(**over)
        L = gpu_gen.make_layer(cfg, 0)
        dims = dims_for(cfg)
        kd = build_kdom(L, dims)
        Kh, Vh = L.k.cpu().pin_memory(), L.v.cpu().pin_memory()
        del L.k, L.v
        torch.cuda.empty_cache()
        ws = _ws(dims, cfg.budget)
        out = torch.empty((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32, device="cuda")
        held = [kd, L.q, L.pos, L.seq_lens, L.dom_fc, out] + ([ws] if ws is not None else [])
        held_bytes = sum(t.numel() * t.element_size() for t in held)
        eq10 = cfg.batch * cfg.n_kv_heads * O.fasa_m_gpu_bytes(1, cfg.context, cfg.head_dim, cfg.n_tip,
                                                               cfg.budget, cfg.elem_bytes)
        assert held_bytes <= eq10
        fasa_decode_step(L.q, L.pos, Kh, Vh, kd, L.dom_fc, L.seq_lens, cfg.budget, out, None, None, ws, dims)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for _ in range(3):
            fasa_decode_step(L.q, L.pos, Kh, Vh, kd, L.dom_fc, L.seq_lens, cfg.budget, out, None, None, ws, dims)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        assert fasa_device_status() == 0
        assert np.all(np.isfinite(out.cpu().numpy()))


def test_step_io_in_host_memory():
    """Zero-copy step I/O: q, pos, lengths, output, indices and counts in
    pinned host memory give the device run's results bit for bit."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_decode_step, fasa_device_status
    cfg = configs.CONFIGS["llama3_8b_ctx32k"].with_(context=8192, batch=2)
    L = gpu_gen.make_layer(cfg, 0)
    L.seq_lens = torch.tensor([8192, 3001], dtype=torch.int32, device="cuda")
    L.pos = L.seq_lens.clone()
    dims = dims_for(cfg)
    kd = build_kdom(L, dims)
    ws = _ws(dims, cfg.budget)
    shape_o = (cfg.batch, cfg.n_q_heads, cfg.head_dim)
    shape_i = (cfg.batch, cfg.n_kv_heads, cfg.budget)
    res = []
    for host in (False, True):
        mk = (lambda t: t.cpu().pin_memory()) if host else (lambda t: t)
        q, pos, lens = mk(L.q), mk(L.pos), mk(L.seq_lens)
        out = mk(torch.full(shape_o, float("nan"), dtype=torch.float32, device="cuda"))
        idx = mk(torch.full(shape_i, -7, dtype=torch.int32, device="cuda"))
        cnt = mk(torch.full(shape_i[:2], -7, dtype=torch.int32, device="cuda"))
        fasa_decode_step(q, pos, L.k, L.v, kd, L.dom_fc, lens, cfg.budget, out, idx, cnt, ws, dims)
        torch.cuda.synchronize()
        assert fasa_device_status() == 0
        res.append((out.cpu(), idx.cpu(), cnt.cpu()))
    L.seq_lens_host = L.seq_lens.cpu().numpy()
    L.pos_host = L.pos.cpu().numpy()
    _check_units(L, cfg, *res[1], units=[(0, 0), (0, 5), (1, 2), (1, 7)])
    for a, b in zip(*res):
        assert torch.equal(a, b)


def _nondom_expected(L, cfg):
    """K^nondom by hand: each token's non-dominant FC pairs in FC order."""
    B, H, T, d = cfg.batch, cfg.n_kv_heads, cfg.context, cfg.head_dim
    k16 = L.k.cpu().view(__import__("torch").int16).numpy().reshape(B, H, T, d // 2, 2)
    out = np.empty((B, H, T, d // 2 - cfg.n_tip, 2), dtype=np.int16)
    for h in range(H):
        nd = np.setdiff1d(np.arange(d // 2), L.dom_fc_host[h])
        out[:, h] = k16[:, h][:, :, nd, :]
    return out


SPLIT_CASES = [("llama3_8b_ctx32k", dict(context=8192, batch=1)),    # single-exchange, list resident
               ("qwen25_7b_b8_ctx16k", dict(context=4096)),            # single-exchange, list streamed
               ("qwen25_7b_b8_ctx16k", dict(context=4096, batch=16))]  # cluster kernel


@pytest.mark.parametrize("name,over", SPLIT_CASES)
def test_split_keys_against_oracle(name, over):
    """FASA-M with split keys: K^nondom and V in host memory, K^dom on the
    GPU.  fasa_build_knondom writes exactly each token's non-dominant pairs;
    the split step selects the same tokens as the whole-key step and its
    output matches the oracle unit by unit."""
    import torch
    from kv_cache_token_tip_gb300 import (dims_for, fasa_build_knondom, fasa_decode_step, fasa_decode_step_split,
                                          fasa_device_status)
    cfg = configs.CONFIGS[name].with_(**over)
    L = gpu_gen.make_layer(cfg, 0)
    dims = dims_for(cfg)
    kd = build_kdom(L, dims)
    ws = _ws(dims, cfg.budget)
    ndp = cfg.head_dim // 2 - cfg.n_tip
    knd = torch.empty((cfg.batch, cfg.n_kv_heads, cfg.context, 2 * ndp), dtype=torch.bfloat16).pin_memory()
    fasa_build_knondom(L.k, L.dom_fc, None, knd, dims)
    torch.cuda.synchronize()
    assert fasa_device_status() == 0
    want = _nondom_expected(L, cfg)
    assert np.array_equal(knd.view(torch.int16).numpy().reshape(want.shape), want)
    Vh = L.v.cpu().pin_memory()
    res = []
    for split in (False, True):
        out = torch.full((cfg.batch, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=torch.float32, device="cuda")
        idx = torch.empty((cfg.batch, cfg.n_kv_heads, cfg.budget), dtype=torch.int32, device="cuda")
        cnt = torch.empty((cfg.batch, cfg.n_kv_heads), dtype=torch.int32, device="cuda")
        if split:
            fasa_decode_step_split(L.q, L.pos, knd, Vh, kd, L.dom_fc, L.seq_lens, cfg.budget, out, idx, cnt, ws, dims)
        else:
            fasa_decode_step(L.q, L.pos, L.k, L.v, kd, L.dom_fc, L.seq_lens, cfg.budget, out, idx, cnt, ws, dims)
        torch.cuda.synchronize()
        assert fasa_device_status() == 0
        res.append((out.cpu(), idx.cpu(), cnt.cpu()))
    assert torch.equal(res[0][1], res[1][1]) and torch.equal(res[0][2], res[1][2])
    _check_units(L, cfg, *res[1])
    P.check_output(res[1][0].numpy(), res[0][0].numpy().astype(np.float64), cfg.dtype)


@pytest.mark.parametrize("name,over,lens", [("llama3_8b_ctx32k", dict(context=8192, batch=2), (8000, 300)),
                                            ("qwen25_7b_b8_ctx16k", dict(context=4096, batch=2), (4000, 1234)),
                                            ("qwen25_7b_b8_ctx16k", dict(context=4096, batch=16),
                                             (4000, 1234, 3500, 4095, 17, 3097, 3098, 2000) * 2)])
def test_split_keys_append_against_oracle(name, over, lens):
    """The append step over split keys: the new token's non-dominant pairs
    land in its k_nondom row (host memory) exactly as fasa_build_knondom
    would write them from the whole rotated key, its dominant pairs in K_dom
    and its value in V exactly as the whole-key append writes them; the
    selection equals the whole-key append step's and the output matches the
    oracle over the appended caches unit by unit."""
    import torch
    from kv_cache_token_tip_gb300 import (dims_for, fasa_build_knondom, fasa_decode_step_append,
                                          fasa_decode_step_append_split, fasa_device_status)
    cfg = configs.CONFIGS[name].with_(**over)
    L = gpu_gen.make_layer(cfg, 0)
    L.seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    dims = dims_for(cfg)
    kd_whole = build_kdom(L, dims)
    kd_split = kd_whole.clone()
    ws = _ws(dims, cfg.budget)
    ndp = cfg.head_dim // 2 - cfg.n_tip
    knd = torch.empty((cfg.batch, cfg.n_kv_heads, cfg.context, 2 * ndp), dtype=torch.bfloat16).pin_memory()
    fasa_build_knondom(L.k, L.dom_fc, None, knd, dims)
    gen = torch.Generator(device="cuda").manual_seed(11)
    shape = (cfg.batch, cfg.n_kv_heads, cfg.head_dim)
    kn = torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
    vn = torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
    Kd, Vd = L.k.clone(), L.v.clone()
    Vh = L.v.cpu().pin_memory()
    res = []
    for split in (False, True):
        out = torch.full((cfg.batch, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=torch.float32, device="cuda")
        idx = torch.empty((cfg.batch, cfg.n_kv_heads, cfg.budget), dtype=torch.int32, device="cuda")
        cnt = torch.empty((cfg.batch, cfg.n_kv_heads), dtype=torch.int32, device="cuda")
        if split:
            fasa_decode_step_append_split(L.q, kn, vn, L.seq_lens, knd, Vh, kd_split, L.dom_fc, cfg.budget, out, idx,
                                          cnt, ws, dims)
        else:
            fasa_decode_step_append(L.q, kn, vn, L.seq_lens, Kd, Vd, kd_whole, L.dom_fc, cfg.budget, out, idx, cnt,
                                    ws, dims)
        torch.cuda.synchronize()
        assert fasa_device_status() == 0
        res.append((out.cpu(), idx.cpu(), cnt.cpu()))
    assert torch.equal(res[0][1], res[1][1]) and torch.equal(res[0][2], res[1][2])
    assert torch.equal(kd_whole, kd_split)
    assert torch.equal(Vd.cpu(), Vh)
    want = _nondom_expected(types.SimpleNamespace(k=Kd, dom_fc_host=L.dom_fc_host), cfg)
    assert np.array_equal(knd.view(torch.int16).numpy().reshape(want.shape), want)
    n = np.asarray(lens)
    Lh = types.SimpleNamespace(cfg=cfg, q=L.q, k=Kd.cpu(), v=Vh, seq_lens_host=n + 1, pos_host=n,
                               dom_fc_host=L.dom_fc_host)
    _check_units(Lh, cfg, *res[1])


def test_split_keys_cover_both_fused_kernels():
    """The cases above run on both fused kernels (the single-exchange kernel
    and the cluster kernel)."""
    from kv_cache_token_tip_gb300 import dims_for, fasa_step_kernel
    kinds = [fasa_step_kernel(dims_for(configs.CONFIGS[n].with_(**o))) for n, o in SPLIT_CASES]
    assert kinds == [1, 1, 0]


def test_split_keys_reject_what_the_layout_cannot_hold():
    """A per-head FC table with unused slots cannot be split: the build and
    the step report FASA_DEV_BAD_INPUT; an N_tip that is not a multiple of 4
    is refused before any launch."""
    import torch
    from kv_cache_token_tip_gb300 import (FASA_DEV_BAD_INPUT, FasaError, dims_for, fasa_build_knondom,
                                          fasa_decode_step_split, fasa_device_status)
    cfg = configs.CONFIGS["llama3_8b_ctx32k_ragged_ntip"].with_(context=4096)
    L = gpu_gen.make_layer(cfg, 0)
    dims = dims_for(cfg)
    kd = build_kdom(L, dims)
    ndp = cfg.head_dim // 2 - cfg.n_tip
    knd = torch.zeros((cfg.batch, cfg.n_kv_heads, cfg.context, 2 * ndp), dtype=torch.bfloat16, device="cuda")
    fasa_device_status()
    fasa_build_knondom(L.k, L.dom_fc, None, knd, dims)
    assert fasa_device_status() & FASA_DEV_BAD_INPUT
    out = torch.empty((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32, device="cuda")
    ws = _ws(dims, cfg.budget)
    fasa_decode_step_split(L.q, L.pos, knd, L.v, kd, L.dom_fc, L.seq_lens, cfg.budget, out, None, None, ws, dims)
    assert fasa_device_status() & FASA_DEV_BAD_INPUT
    odd = dims_for(configs.CONFIGS["llama3_8b_ctx32k"].with_(context=4096, n_tip=6))
    with pytest.raises(FasaError):
        fasa_decode_step_split(L.q, L.pos, knd, L.v, kd, L.dom_fc, L.seq_lens, cfg.budget, out, None, None, ws, odd)
