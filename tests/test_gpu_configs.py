"""The fused decode step at the full sizes of the five workloads, against the
fp64 oracle on the same stored bytes (GPU).

Every (batch, KV head) unit is checked where the oracle finishes in seconds;
the 32-layer ragged workload checks a fixed sample of units in every layer.
The launch configuration is the one the benchmark times (automatic cluster
size, workspace from fasa_workspace_size).
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


def _run_step(L, cfg, dims):
    import torch
    from kv_cache_token_tip_gb300 import fasa_decode_step, fasa_device_status, fasa_workspace_size
    kd = build_kdom(L, dims)
    B, Hq, H, d, k = cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.budget
    ws_bytes = fasa_workspace_size(dims, k)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda") if ws_bytes else None
    out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.empty((B, H, k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B, H), dtype=torch.int32, device="cuda")
    fasa_decode_step(L.q, L.pos, L.k, L.v, kd, L.dom_fc, L.seq_lens, k, out, idx, cnt, ws, dims)
    assert fasa_device_status() == 0
    del kd
    return out.cpu().numpy(), idx.cpu().numpy(), cnt.cpu().numpy(), ws_bytes


def _check_unit(L, cfg, o, ix, cn, b, h):
    k, G = cfg.budget, cfg.group
    ref = oracle_unit(L, b, h, k)
    Lb = int(L.seq_lens_host[b])
    assert cn[b, h] == min(k, Lb)
    mine = ix[b, h, :cn[b, h]]
    P.check_selection(mine, ref["scores"], k)
    fac_ref = O.focused_attention_unit(ref["q_rot"], ref["K"], ref["V"], mine)
    P.check_output(o[b, h * G:(h + 1) * G], fac_ref, cfg.dtype)
    if np.array_equal(mine, ref["idx"]):
        P.check_output(o[b, h * G:(h + 1) * G], ref["out"], cfg.dtype)


@pytest.mark.parametrize("name", ["tiny_fp32_ctx1k", "llama3_8b_ctx32k", "qwen25_7b_b8_ctx16k",
                                  "llama3_8b_b4_ctx128k"])
def test_full_workload(name):
    from kv_cache_token_tip_gb300 import dims_for
    cfg = configs.CONFIGS[name]
    L = gpu_gen.make_layer(cfg, 0)
    dims = dims_for(cfg)
    o, ix, cn, ws = _run_step(L, cfg, dims)
    if name == "llama3_8b_b4_ctx128k":
        assert ws > 0   # scores of a 32K-token CTA range go to the caller's workspace
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            _check_unit(L, cfg, o, ix, cn, b, h)


def test_mistral_32_layers_ragged():
    """All 32 layers of the ragged batch-32 workload run; a fixed sample of
    (sequence, KV head) units of every layer is checked against the oracle."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for
    cfg = configs.CONFIGS["mistral_7b_l32_b32_ragged"]
    dims = dims_for(cfg)
    q, k, v = gpu_gen.alloc_layer(cfg)
    sample = [(0, 0), (7, 3), (15, 5), (31, 7)]
    from workload import synth
    lens = torch.from_numpy(synth.seq_lens(cfg)).cuda()
    for layer in range(cfg.layers):
        gpu_gen.fill_layer(cfg, layer, q, k, v)
        dom = torch.from_numpy(synth.dominant_fcs(cfg, layer)).cuda()
        L = gpu_gen.DeviceLayer(cfg, q, k, v, dom, lens, lens.clone())
        o, ix, cn, _ = _run_step(L, cfg, dims)
        assert np.all(np.isfinite(o))
        assert np.array_equal(cn, np.minimum(cfg.budget, L.seq_lens_host)[:, None].repeat(cfg.n_kv_heads, 1))
        for (b, h) in sample:
            _check_unit(L, cfg, o, ix, cn, b, h)


def test_dense_full_size_sample():
    """Dense decode attention over all 32K cached tokens (the sparse-vs-dense
    baseline) on a sample of heads."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_apply_rope_q, fasa_dense_attention
    cfg = configs.CONFIGS["llama3_8b_ctx32k"]
    L = gpu_gen.make_layer(cfg, 0)
    dims = dims_for(cfg)
    q_rot = torch.empty((1, 32, 128), dtype=torch.float32, device="cuda")
    fasa_apply_rope_q(L.q, L.pos, q_rot, dims)
    out = torch.empty_like(q_rot)
    fasa_dense_attention(q_rot, L.k, L.v, L.seq_lens, out, dims)
    o = out.cpu().numpy()
    for h in (0, 5):
        ref = oracle_unit(L, 0, h, cfg.budget)
        dense = O.focused_attention_unit(ref["q_rot"], ref["K"], ref["V"], np.arange(cfg.context))
        P.check_output(o[0, 4 * h:4 * h + 4], dense, "bf16")


@pytest.mark.parametrize("name", ["llama3_8b_ctx32k", "qwen25_7b_b8_ctx16k", "llama3_8b_b4_ctx128k"])
def test_step_without_index_output(name):
    """The step as the benchmark times it -- no idx_out / count_out -- gives
    bit for bit the output of the step that also writes the indices (whose
    selection and output the full-workload test checks against the oracle);
    a sample of units is checked against the oracle directly."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_decode_step, fasa_device_status, fasa_workspace_size
    cfg = configs.CONFIGS[name]
    L = gpu_gen.make_layer(cfg, 0)
    dims = dims_for(cfg)
    o_idx, ix, cn, _ = _run_step(L, cfg, dims)
    kd = build_kdom(L, dims)
    ws_bytes = fasa_workspace_size(dims, cfg.budget)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda") if ws_bytes else None
    out = torch.full((cfg.batch, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    fasa_decode_step(L.q, L.pos, L.k, L.v, kd, L.dom_fc, L.seq_lens, cfg.budget, out, None, None, ws, dims)
    assert fasa_device_status() == 0
    o = out.cpu().numpy()
    assert np.array_equal(o, o_idx)
    for (b, h) in [(0, 0), (cfg.batch - 1, cfg.n_kv_heads - 1)]:
        _check_unit(L, cfg, o, ix, cn, b, h)


@pytest.mark.parametrize("over", [dict(dtype="bf16", context=8192, budget=256),
                                  dict(dtype="bf16", context=8192, budget=256, batch=3)])
def test_head_dim_64_bf16(over):
    """bf16 with head_dim 64 (the tiny workload's shape, stored in bf16 at
    8K tokens): the single-exchange kernel at batch 1 (clusters of 16) and
    the cluster kernel or the single-exchange kernel at batch 3, every unit
    against the oracle."""
    from kv_cache_token_tip_gb300 import dims_for, fasa_step_kernel
    cfg = configs.CONFIGS["tiny_fp32_ctx1k"].with_(**over)
    L = gpu_gen.make_layer(cfg, 0)
    dims = dims_for(cfg)
    if cfg.batch == 1:
        assert fasa_step_kernel(dims) == 1
    o, ix, cn, _ = _run_step(L, cfg, dims)
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            _check_unit(L, cfg, o, ix, cn, b, h)
