"""Variants of the step the FASA pages describe (GPU): per-head N_tip
("Layer-wise and head-wise N_tip optimization"), every FC dominant (the
pages' "Oracle" selection through the same kernels) and per-layer budgets.

A head keeps the entries of its dominant-FC row before the first negative
one; the step reads only those planes of K_dom.  Each case is checked
against the fp64 oracle, and the ragged step bit for bit against uniform
launches that give every head the same count.
"""

import numpy as np
import pytest

import oracle as O
from tests import parity as P
from tests.gpu_util import build_kdom, ensure_built, oracle_unit
from workload import configs, gpu_gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    ensure_built()


def _run(L, cfg, dims, kd, budget, dom=None):
    import torch
    from kv_cache_token_tip_gb300 import fasa_decode_step, fasa_device_status, fasa_workspace_size
    n = fasa_workspace_size(dims, budget)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda") if n else None
    out = torch.full((cfg.batch, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.empty((cfg.batch, cfg.n_kv_heads, budget), dtype=torch.int32, device="cuda")
    cnt = torch.empty((cfg.batch, cfg.n_kv_heads), dtype=torch.int32, device="cuda")
    fasa_decode_step(L.q, L.pos, L.k, L.v, kd, L.dom_fc if dom is None else dom, L.seq_lens, budget, out, idx, cnt,
                     ws, dims)
    assert fasa_device_status() == 0
    return out.cpu().numpy(), idx.cpu().numpy(), cnt.cpu().numpy()


def _check_layer(L, cfg, res, budget):
    out, idx, cnt = res
    G = cfg.group
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            ref = oracle_unit(L, b, h, budget)
            assert cnt[b, h] == min(budget, int(L.seq_lens_host[b]))
            mine = idx[b, h, :cnt[b, h]]
            P.check_selection(mine, ref["scores"], budget)
            sel_out = O.focused_attention_unit(ref["q_rot"], ref["K"], ref["V"], mine)
            P.check_output(out[b, h * G:(h + 1) * G], sel_out, cfg.dtype)


def _layer(name, **over):
    cfg = configs.CONFIGS[name].with_(**over)
    L = gpu_gen.make_layer(cfg, 0)
    return cfg, L


def test_ragged_ntip_against_oracle():
    import torch
    from kv_cache_token_tip_gb300 import dims_for
    cfg, L = _layer("llama3_8b_ctx32k_ragged_ntip", context=8192, batch=2)
    L.seq_lens = torch.tensor([8192, 5000], dtype=torch.int32, device="cuda")
    L.pos = L.seq_lens.clone()
    L.seq_lens_host, L.pos_host = np.array([8192, 5000]), np.array([8192, 5000])
    assert sorted(set((L.dom_fc_host >= 0).sum(axis=1).tolist())) == sorted(set(cfg.n_tip_per_head))
    dims = dims_for(cfg)
    kd = build_kdom(L, dims)
    _check_layer(L, cfg, _run(L, cfg, dims, kd, cfg.budget), cfg.budget)


@pytest.mark.parametrize("cluster", [4, 12])
def test_ragged_heads_equal_uniform_launches(cluster):
    """Each head of the ragged step gives bit for bit what a launch giving
    every head that head's count gives it (same FCs, same cluster size)."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for
    cfg, L = _layer("llama3_8b_ctx32k_ragged_ntip", context=8192, batch=2)
    dims = dims_for(cfg, cluster_ctas=cluster)
    kd = build_kdom(L, dims)
    out, idx, cnt = _run(L, cfg, dims, kd, cfg.budget)
    G = cfg.group
    dom_host = L.dom_fc_host
    for n_h in sorted(set(cfg.n_tip_per_head)):
        heads = [h for h in range(cfg.n_kv_heads) if cfg.n_tip_per_head[h] == n_h]
        # every head gets n_h FCs: its own set where it has n_h, else any n_h FCs
        dom = np.stack([dom_host[h, :n_h] if cfg.n_tip_per_head[h] >= n_h else np.arange(n_h)
                        for h in range(cfg.n_kv_heads)]).astype(np.int32)
        dom_d = torch.from_numpy(dom).cuda()
        d_u = dims_for(cfg, cluster_ctas=cluster, n_tip=n_h)
        kd_u = torch.empty((cfg.batch, cfg.n_kv_heads, cfg.context // 64, n_h, 64, 2), dtype=L.k.dtype,
                           device="cuda")
        from kv_cache_token_tip_gb300 import fasa_build_kdom
        fasa_build_kdom(L.k, dom_d, None, kd_u, d_u)
        o2, i2, c2 = _run(L, cfg, d_u, kd_u, cfg.budget, dom=dom_d)
        for h in heads:
            assert np.array_equal(cnt[:, h], c2[:, h])
            assert np.array_equal(idx[:, h], i2[:, h])
            assert np.array_equal(out[:, h * G:(h + 1) * G], o2[:, h * G:(h + 1) * G])


def test_ragged_kdom_and_append_touch_only_used_planes():
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_decode_step_append, fasa_device_status
    cfg, L = _layer("llama3_8b_ctx32k_ragged_ntip", context=4096, batch=2)
    L.seq_lens = torch.tensor([3000, 17], dtype=torch.int32, device="cuda")
    dims = dims_for(cfg)
    kd = torch.full((cfg.batch, cfg.n_kv_heads, cfg.context // 64, cfg.n_tip, 64, 2), 7.0, dtype=L.k.dtype,
                    device="cuda")
    from kv_cache_token_tip_gb300 import fasa_build_kdom
    fasa_build_kdom(L.k, L.dom_fc, None, kd, dims)
    gen = torch.Generator(device="cuda").manual_seed(3)
    shape = (cfg.batch, cfg.n_kv_heads, cfg.head_dim)
    kn = torch.randn(shape, generator=gen, device="cuda").to(L.k.dtype)
    vn = torch.randn(shape, generator=gen, device="cuda").to(L.k.dtype)
    out = torch.empty((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32, device="cuda")
    from kv_cache_token_tip_gb300 import fasa_workspace_size
    n = fasa_workspace_size(dims, cfg.budget)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda") if n else None
    fasa_decode_step_append(L.q, kn, vn, L.seq_lens, L.k, L.v, kd, L.dom_fc, cfg.budget, out, None, None, ws,
                            dims)
    assert fasa_device_status() == 0
    kdh = kd.float().cpu().numpy()
    K = L.k.float().cpu().numpy()
    lens = [3000, 17]
    for h in range(cfg.n_kv_heads):
        n_h = cfg.n_tip_per_head[h]
        for j in range(cfg.n_tip):
            plane = kdh[:, h, :, j].reshape(cfg.batch, cfg.context, 2)
            if j < n_h:
                i = L.dom_fc_host[h, j]
                for b in range(cfg.batch):
                    t = lens[b] + 1   # the appended token included
                    assert np.array_equal(plane[b, :t], K[b, h, :t, 2 * i:2 * i + 2])
            else:
                assert np.all(plane == 7.0)   # unused slots untouched


def test_oracle_k_against_oracle():
    """Every FC dominant: TIP scores are the group-summed logits, so the
    selection is the pages' Oracle top-k."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for
    cfg, L = _layer("llama3_8b_ctx32k_oraclek", context=8192, batch=2)
    assert np.array_equal(L.dom_fc_host, np.tile(np.arange(64), (cfg.n_kv_heads, 1)))
    dims = dims_for(cfg)
    kd = build_kdom(L, dims)
    res = _run(L, cfg, dims, kd, cfg.budget)
    _check_layer(L, cfg, res, cfg.budget)
    # the selection is the top-k of the full logits (rotated query . key)
    G = cfg.group
    for b in range(cfg.batch):
        for h in (0, 5):
            ref = oracle_unit(L, b, h, cfg.budget)
            logits = ref["K"] @ ref["q_rot"].sum(axis=0)
            P.check_selection(res[1][b, h, :res[2][b, h]], logits, cfg.budget)


def test_pyramid_budgets_per_layer():
    from kv_cache_token_tip_gb300 import dims_for
    cfg = configs.CONFIGS["mistral_7b_l32_b32_pyramid"].with_(context=4096, batch=2, ragged=(1000, 4096))
    dims = dims_for(cfg)
    for layer in (0, 13, 31):
        L = gpu_gen.make_layer(cfg, layer)
        kd = build_kdom(L, dims)
        budget = cfg.layer_budget(layer)
        _check_layer(L, cfg, _run(L, cfg, dims, kd, budget), budget)
