"""fasa_decode_step_append: the decode step with the new token's cache
maintenance fused in (GPU).

The new token's key is rotated by its position len and stored, with its value
and its dominant FCs, at index len; the step then attends over len + 1
tokens with the query at position len.  Checked against the fp64 oracle on
the bytes the library stored, and bit for bit against the same step done in
separate launches (cache rows, fasa_append_kdom, fasa_decode_step).
"""

import numpy as np
import pytest

import oracle as O
from tests import parity as P
from tests.gpu_util import build_kdom, ensure_built
from workload import configs, gpu_gen, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    ensure_built()


def _stored_device(x64, dtype):
    import torch
    st = synth.store(x64, dtype)
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(st)).cuda()
    return torch.from_numpy(np.ascontiguousarray(st).view(np.int16)).cuda().view(torch.bfloat16)


def _case(cfg, lens, seed):
    """A layer of `cfg` whose sequences hold `lens` tokens, plus a new token
    per (batch, KV head)."""
    import torch
    L = gpu_gen.make_layer(cfg, 0)
    L.seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    L.seq_lens_host = np.asarray(lens, dtype=np.int64)
    rng = np.random.default_rng(seed)
    shape = (cfg.batch, cfg.n_kv_heads, cfg.head_dim)
    k_new = _stored_device(rng.standard_normal(shape) * 2.0, cfg.dtype)
    v_new = _stored_device(rng.standard_normal(shape), cfg.dtype)
    return L, k_new, v_new


def _run_append(L, cfg, dims, k_new, v_new, kd, budget):
    import torch
    from kv_cache_token_tip_gb300 import fasa_decode_step_append, fasa_workspace_size
    ws_bytes = fasa_workspace_size(dims, budget)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda") if ws_bytes else None
    out = torch.full((cfg.batch, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.empty((cfg.batch, cfg.n_kv_heads, budget), dtype=torch.int32, device="cuda")
    cnt = torch.empty((cfg.batch, cfg.n_kv_heads), dtype=torch.int32, device="cuda")
    fasa_decode_step_append(L.q, k_new, v_new, L.seq_lens, L.k, L.v, kd, L.dom_fc, budget, out, idx, cnt, ws, dims)
    return out, idx, cnt, ws


def _check_against_oracle(L, cfg, k_new, v_new, kd, out, idx, cnt, budget):
    import torch
    G = cfg.group
    lens = L.seq_lens_host
    o, ix, cn = out.cpu().numpy(), idx.cpu().numpy(), cnt.cpu().numpy()
    kn = P.host_f64(k_new, cfg.dtype)
    q = P.host_f64(L.q, cfg.dtype)
    # the stored key: fp32 rotation (sin/cos of the angle to ~1e-7 of the FC
    # pair's norm) rounded to the storage type (1 ulp of the component in bf16)
    one_ulp = 2.0 ** -7 if cfg.dtype == "bf16" else 0.0
    for b in range(cfg.batch):
        t = int(lens[b])
        Kb = P.host_f64(L.k[b, :, :t + 1], cfg.dtype)
        Vb = P.host_f64(L.v[b, :, :t + 1], cfg.dtype)
        # the stored value row is the new value, bit for bit
        assert torch.equal(L.v[b, :, t], v_new[b])
        # the stored key row is the new key rotated by t, to the storage precision
        ref = O.rope_rotate(kn[b], t, cfg.rope_theta)
        pair = np.repeat(np.hypot(ref[:, 0::2], ref[:, 1::2]), 2, axis=1)
        assert np.all(np.abs(Kb[:, t] - ref) <= one_ulp * np.abs(ref) + 1e-6 * pair)
        # the dominant FCs of the stored key sit in K_dom at t
        for h in range(cfg.n_kv_heads):
            for j, i in enumerate(L.dom_fc_host[h]):
                assert torch.equal(kd[b, h, t // 64, j, t % 64], L.k[b, h, t, 2 * i:2 * i + 2])
        q_rot = O.apply_rope_q(q[b:b + 1], np.array([t]), cfg.rope_theta)[0]
        for h in range(cfg.n_kv_heads):
            qg = q_rot[h * G:(h + 1) * G]
            scores = O.tip_scores_unit(qg, Kb[h], L.dom_fc_host[h])
            ref_idx = O.topk_select_unit(scores, budget)
            assert cn[b, h] == min(budget, t + 1)
            mine = ix[b, h, :cn[b, h]]
            P.check_selection(mine, scores, budget)
            P.check_output(o[b, h * G:(h + 1) * G], O.focused_attention_unit(qg, Kb[h], Vb[h], mine), cfg.dtype)
            if np.array_equal(mine, ref_idx):
                P.check_output(o[b, h * G:(h + 1) * G], O.focused_attention_unit(qg, Kb[h], Vb[h], ref_idx),
                               cfg.dtype)


CASES = [
    # (config, overrides, lengths before the step)
    ("llama3_8b_ctx32k", dict(context=8192, batch=3), [5000, 0, 8191]),
    ("qwen25_7b_b8_ctx16k", dict(context=4096, batch=3, budget=700), [4095, 1234, 100]),
    ("tiny_fp32_ctx1k", dict(batch=2), [1023, 63]),
]


@pytest.mark.parametrize("name,over,lens", CASES, ids=[c[0] for c in CASES])
def test_append_step_against_oracle(name, over, lens):
    from kv_cache_token_tip_gb300 import dims_for, fasa_device_status
    cfg = configs.CONFIGS[name].with_(**over)
    L, k_new, v_new = _case(cfg, lens, 7)
    dims = dims_for(cfg)
    kd = build_kdom(L, dims)
    out, idx, cnt, _ = _run_append(L, cfg, dims, k_new, v_new, kd, cfg.budget)
    assert fasa_device_status() == 0
    _check_against_oracle(L, cfg, k_new, v_new, kd, out, idx, cnt, cfg.budget)


@pytest.mark.parametrize("cluster", [0, 1, 3, 8])
def test_append_step_equals_separate_launches(cluster):
    """Bit for bit the result of writing the rows, fasa_append_kdom and a
    plain fasa_decode_step over len + 1 tokens with the query at len (the
    fused path scores the new token exactly as TIP scores a streamed one)."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_append_kdom, fasa_decode_step, fasa_device_status
    cfg = configs.CONFIGS["llama3_8b_ctx32k"].with_(context=8192, batch=2)
    lens = [6000, 129]
    L, k_new, v_new = _case(cfg, lens, 11)
    dims = dims_for(cfg, cluster_ctas=cluster)
    kd = build_kdom(L, dims)
    K0, V0, kd0 = L.k.clone(), L.v.clone(), kd.clone()
    out, idx, cnt, ws = _run_append(L, cfg, dims, k_new, v_new, kd, cfg.budget)
    assert fasa_device_status() == 0
    # the same step in separate launches, from the rows the fused step stored
    rows = torch.stack([L.k[b, :, lens[b]] for b in range(cfg.batch)])
    for b in range(cfg.batch):
        K0[b, :, lens[b]] = L.k[b, :, lens[b]]
        V0[b, :, lens[b]] = L.v[b, :, lens[b]]
    fasa_append_kdom(rows, L.dom_fc, L.seq_lens, kd0, dims)
    lens1 = L.seq_lens + 1
    out2 = torch.full_like(out, float("nan"))
    idx2, cnt2 = torch.empty_like(idx), torch.empty_like(cnt)
    fasa_decode_step(L.q, L.seq_lens, K0, V0, kd0, L.dom_fc, lens1, cfg.budget, out2, idx2, cnt2, ws, dims)
    assert fasa_device_status() == 0
    assert torch.equal(kd, kd0) and torch.equal(L.k, K0) and torch.equal(L.v, V0)
    assert torch.equal(idx, idx2) and torch.equal(cnt, cnt2)
    assert torch.equal(out, out2)


def test_append_decode_loop_keeps_kdom_in_step():
    """Four steps of a decode loop (the caller advancing the lengths): K_dom
    stays equal to the K_dom rebuilt from the final cache, and the last step
    matches the oracle."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_device_status
    cfg = configs.CONFIGS["llama3_8b_ctx32k"].with_(context=4096, batch=2)
    L, k_new, v_new = _case(cfg, [3000, 62], 5)
    dims = dims_for(cfg)
    kd = build_kdom(L, dims)
    for step in range(4):
        rng = np.random.default_rng(100 + step)
        shape = (cfg.batch, cfg.n_kv_heads, cfg.head_dim)
        k_new = _stored_device(rng.standard_normal(shape) * 2.0, cfg.dtype)
        v_new = _stored_device(rng.standard_normal(shape), cfg.dtype)
        out, idx, cnt, _ = _run_append(L, cfg, dims, k_new, v_new, kd, cfg.budget)
        assert fasa_device_status() == 0
        if step < 3:
            L.seq_lens += 1
            L.seq_lens_host = L.seq_lens_host + 1
    _check_against_oracle(L, cfg, k_new, v_new, kd, out, idx, cnt, cfg.budget)
    # K_dom was built over the whole cache and each step rewrote its token:
    # it equals the K_dom rebuilt from the final cache everywhere
    assert torch.equal(kd, build_kdom(L, dims))


def test_append_into_a_full_cache_is_reported():
    """A sequence whose cache is full cannot take the token: the device status
    reports bad input and the other sequences still step normally."""
    from kv_cache_token_tip_gb300 import dims_for, fasa_device_status
    cfg = configs.CONFIGS["llama3_8b_ctx32k"].with_(context=4096, batch=2)
    L, k_new, v_new = _case(cfg, [4096, 1000], 3)
    dims = dims_for(cfg)
    kd = build_kdom(L, dims)
    out, idx, cnt, _ = _run_append(L, cfg, dims, k_new, v_new, kd, cfg.budget)
    assert fasa_device_status() & 1
    o = out.cpu().numpy()
    assert np.all(np.isfinite(o))
    assert np.all(cnt.cpu().numpy()[1] == cfg.budget)
