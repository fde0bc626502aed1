"""Per-stage parity of the CUDA library against the fp64 oracle (GPU).

Every comparison runs on the stored bytes that were fed to the GPU.  Sizes are
ones the oracle finishes in seconds but that still span several TIP tiles,
several CTAs of a cluster and a ragged tail.
"""

import numpy as np
import pytest

import oracle as O
from tests import parity as P
from tests.gpu_util import build_kdom, ensure_built, oracle_unit
from workload import configs, gpu_gen, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    ensure_built()


def _cfg(name, **kw):
    return configs.CONFIGS[name].with_(**kw)


def _layer(cfg, lens=None, layer=0):
    import torch
    L = gpu_gen.make_layer(cfg, layer)
    if lens is not None:
        L.seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
        L.pos = L.seq_lens.clone()
        L.seq_lens_host = np.asarray(lens, dtype=np.int32)
        L.pos_host = L.seq_lens_host.copy()
    return L


SMALL = [
    ("tiny_fp32_ctx1k", dict()),
    ("llama3_8b_ctx32k", dict(context=4096, batch=2)),
    ("qwen25_7b_b8_ctx16k", dict(context=2048, batch=2, budget=389)),
]


def test_library_loads_and_version():
    from kv_cache_token_tip_gb300 import lib
    assert lib().fasa_version() >= 100


@pytest.mark.parametrize("name,kw", SMALL)
def test_apply_rope_q(name, kw):
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_apply_rope_q
    cfg = _cfg(name, **kw)
    L = _layer(cfg)
    dims = dims_for(cfg)
    q_rot = torch.empty(L.q.shape, dtype=torch.float32, device="cuda")
    fasa_apply_rope_q(L.q, L.pos, q_rot, dims)
    ref = O.apply_rope_q(P.host_f64(L.q, cfg.dtype), L.pos_host, cfg.rope_theta)
    got = q_rot.cpu().numpy().astype(np.float64)
    # fp32 rotation of exactly represented inputs: error ~1e-7 of the FC norm
    norm = np.sqrt(ref[..., 0::2] ** 2 + ref[..., 1::2] ** 2).repeat(2, axis=-1)
    assert np.all(np.abs(got - ref) <= 2e-6 * np.maximum(norm, 1e-30) + 1e-30)


@pytest.mark.parametrize("name,kw", SMALL)
def test_build_and_append_kdom_bit_exact(name, kw):
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_append_kdom, fasa_build_kdom
    cfg = _cfg(name, **kw)
    L = _layer(cfg)
    dims = dims_for(cfg)
    kd = build_kdom(L, dims)
    ref = O.build_kdom(L.k.cpu().numpy() if cfg.dtype == "f32" else
                       L.k.view(torch.int16).cpu().numpy(), L.dom_fc_host)
    got = kd.cpu().numpy() if cfg.dtype == "f32" else kd.view(torch.int16).cpu().numpy()
    assert np.array_equal(got, ref)

    def fc_major(a):   # [B,H,T/64,n,64,2] -> [B,H,n,T,2]
        B_, H_, nb, n_, kb, _ = a.shape
        return a.transpose(0, 1, 3, 2, 4, 5).reshape(B_, H_, n_, nb * kb, 2)
    ref = fc_major(ref)
    # ragged build touches only tau < len
    lens = np.array([max(1, cfg.context - 37 * (b + 1)) for b in range(cfg.batch)], dtype=np.int32)
    kd2 = torch.zeros_like(kd)
    fasa_build_kdom(L.k, L.dom_fc, torch.from_numpy(lens).cuda(), kd2, dims)
    g2 = fc_major(kd2.cpu().numpy() if cfg.dtype == "f32" else kd2.view(torch.int16).cpu().numpy())
    for b in range(cfg.batch):
        assert np.array_equal(g2[b, :, :, :lens[b]], ref[b, :, :, :lens[b]])
        assert not np.any(g2[b, :, :, lens[b]:])
    # append one token per sequence at slot len_b
    k_new = torch.randn((cfg.batch, cfg.n_kv_heads, cfg.head_dim), device="cuda").to(L.k.dtype)
    slots = torch.from_numpy(np.minimum(lens, cfg.context - 1)).cuda()
    fasa_append_kdom(k_new, L.dom_fc, slots, kd2, dims)
    g3 = fc_major(kd2.cpu().numpy() if cfg.dtype == "f32" else kd2.view(torch.int16).cpu().numpy())
    kn = k_new.cpu().numpy() if cfg.dtype == "f32" else k_new.view(torch.int16).cpu().numpy()
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            for j, i in enumerate(L.dom_fc_host[h]):
                assert np.array_equal(g3[b, h, j, slots[b].item()], kn[b, h, 2 * i:2 * i + 2])


@pytest.mark.parametrize("name,kw", SMALL)
def test_tip_topk_fac_stages(name, kw):
    """TIP scores, top-k on the library's own fp32 scores (bit-exact against the
    oracle's TopK-I on the same values), FAC and dense attention."""
    import torch
    from kv_cache_token_tip_gb300 import (dims_for, fasa_apply_rope_q, fasa_dense_attention,
                                          fasa_focused_attention, fasa_tip_score, fasa_topk_select)
    cfg = _cfg(name, **kw)
    T = cfg.context
    lens = [T - 5 - 333 * b for b in range(cfg.batch)]
    L = _layer(cfg, lens)
    dims = dims_for(cfg)
    kd = build_kdom(L, dims)
    B, Hq, H, d, k = cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.budget
    q_rot = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    fasa_apply_rope_q(L.q, L.pos, q_rot, dims)
    scores = torch.full((B, H, T), float("nan"), dtype=torch.float32, device="cuda")
    fasa_tip_score(q_rot, kd, L.dom_fc, L.seq_lens, scores, dims)
    idx = torch.empty((B, H, k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B, H), dtype=torch.int32, device="cuda")
    fasa_topk_select(scores, L.seq_lens, k, idx, cnt, dims)
    out = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
    fasa_focused_attention(q_rot, L.k, L.v, L.seq_lens, idx, cnt, k, out, dims)
    dense = torch.empty_like(out)
    fasa_dense_attention(q_rot, L.k, L.v, L.seq_lens, dense, dims)
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    ix = idx.cpu().numpy()
    cn = cnt.cpu().numpy()
    o = out.cpu().numpy()
    dn = dense.cpu().numpy()
    G = cfg.group
    for b in range(B):
        for h in range(H):
            ref = oracle_unit(L, b, h, k)
            Lb = lens[b]
            P.check_scores(sc[b, h, :Lb], ref["scores"])
            # selection on the library's fp32 scores: must be exactly TopK-I
            mine = O.topk_select_unit(sc[b, h, :Lb].astype(np.float64), k)
            assert cn[b, h] == min(k, Lb)
            assert np.array_equal(ix[b, h, :cn[b, h]], mine)
            assert np.all(ix[b, h, cn[b, h]:] == -1)
            P.check_selection(ix[b, h, :cn[b, h]], ref["scores"], k)
            fac_ref = O.focused_attention_unit(ref["q_rot"], ref["K"], ref["V"], mine)
            P.check_output(o[b, h * G:(h + 1) * G], fac_ref, cfg.dtype)
            dense_ref = O.focused_attention_unit(ref["q_rot"], ref["K"], ref["V"], np.arange(Lb))
            P.check_output(dn[b, h * G:(h + 1) * G], dense_ref, cfg.dtype)


def _topk_case(scores_np, lens, k, C=0):
    import torch
    from kv_cache_token_tip_gb300 import FasaDims, fasa_topk_select
    B, H, T = scores_np.shape
    dims = FasaDims(B, H, H, 128, T, 8, 1, C, 1e4)
    s = torch.from_numpy(scores_np.astype(np.float32)).cuda()
    ln = torch.tensor(lens, dtype=torch.int32, device="cuda")
    idx = torch.empty((B, H, k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B, H), dtype=torch.int32, device="cuda")
    fasa_topk_select(s, ln, k, idx, cnt, dims)
    ix, cn = idx.cpu().numpy(), cnt.cpu().numpy()
    for b in range(B):
        for h in range(H):
            ref = O.topk_select_unit(scores_np[b, h, :lens[b]].astype(np.float32).astype(np.float64), k)
            assert cn[b, h] == ref.shape[0]
            assert np.array_equal(ix[b, h, :cn[b, h]], ref), (b, h)


@pytest.mark.parametrize("C", [0, 1, 2, 3, 8, 16])
def test_topk_ties_and_modes(C):
    """Bit-exact TopK-I on adversarial scores, for several cluster sizes:
    all-equal (resolved by token order), few distinct values, signed zeros,
    scores sharing their top bits (several radix passes before candidates fit),
    exact-fill buckets and heavy ties at the threshold."""
    rng = np.random.default_rng(0)
    T = 32768
    cases = []
    cases.append(np.zeros((1, 2, T)))                                       # all equal
    cases.append(rng.integers(-2, 3, size=(1, 2, T)).astype(np.float64))    # 5 values
    z = np.where(rng.random((1, 2, T)) < 0.5, 0.0, -0.0)
    z[0, 0, ::97] = 1.0
    cases.append(z)                                                          # +-0
    cases.append(1.0 + rng.random((1, 2, T)) * 2.0 ** -12)                   # shared top bits
    cases.append(rng.standard_normal((1, 2, T)) * 1e3)
    v = np.repeat(np.arange(T // 64, dtype=np.float64), 64)[None, None, :].repeat(2, 1)
    cases.append(v)                                                          # blocks of 64 ties
    for s in cases:
        for k in (1, 64, 256, 1000, 5000):
            _topk_case(s, [T], k, C)
            _topk_case(s, [T - 3], k, C)


def test_topk_ragged_lengths():
    rng = np.random.default_rng(1)
    T = 4096
    lens = [1, 2, 63, 64, 65, 4095, 4096, 100]
    s = rng.standard_normal((len(lens), 3, T))
    s[:, :, ::5] = 0.25   # ties
    for k in (1, 64, 65, 4096):
        _topk_case(s, lens, k)


@pytest.mark.parametrize("C", [0, 1, 2, 4, 8, 16])
def test_decode_step_cluster_sizes(C):
    """The fused step against the oracle for every cluster size."""
    _decode_step_check(_cfg("llama3_8b_ctx32k", context=8192, batch=1), [8192], C)


@pytest.mark.parametrize("name,kw,lens", [
    ("tiny_fp32_ctx1k", dict(), [1024]),
    ("tiny_fp32_ctx1k", dict(batch=3), [1, 64, 999]),
    ("llama3_8b_ctx32k", dict(context=4096, batch=4), [4096, 257, 256, 4093]),
    ("qwen25_7b_b8_ctx16k", dict(context=2048, batch=3, budget=389), [2048, 390, 1500]),
    ("llama3_8b_b4_ctx128k", dict(context=8192, batch=2), [8192, 5000]),
])
def test_decode_step(name, kw, lens):
    _decode_step_check(_cfg(name, **kw), lens, 0)


def _decode_step_check(cfg, lens, C):
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_decode_step, fasa_device_status, fasa_workspace_size
    L = _layer(cfg, lens)
    dims = dims_for(cfg, cluster_ctas=C)
    kd = build_kdom(L, dims)
    B, Hq, H, d, k = cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.budget
    ws_bytes = fasa_workspace_size(dims, k)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.empty((B, H, k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B, H), dtype=torch.int32, device="cuda")
    fasa_decode_step(L.q, L.pos, L.k, L.v, kd, L.dom_fc, L.seq_lens, k, out, idx, cnt,
                     ws if ws_bytes else None, dims)
    assert fasa_device_status() == 0
    o, ix, cn = out.cpu().numpy(), idx.cpu().numpy(), cnt.cpu().numpy()
    G = cfg.group
    for b in range(B):
        for h in range(H):
            ref = oracle_unit(L, b, h, k)
            assert cn[b, h] == min(k, lens[b])
            mine = ix[b, h, :cn[b, h]]
            P.check_selection(mine, ref["scores"], k)
            fac_ref = O.focused_attention_unit(ref["q_rot"], ref["K"], ref["V"], mine)
            P.check_output(o[b, h * G:(h + 1) * G], fac_ref, cfg.dtype)
            if np.array_equal(mine, ref["idx"]):
                P.check_output(o[b, h * G:(h + 1) * G], ref["out"], cfg.dtype)


def test_all_fcs_full_budget_is_dense():
    """With every FC dominant and budget >= len the fused step is dense
    attention of the rotated query, and the TIP scores are the summed logits."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_apply_rope_q, fasa_decode_step, fasa_tip_score
    cfg = _cfg("tiny_fp32_ctx1k", n_tip=32, budget=1024)
    L = _layer(cfg)
    L.dom_fc = torch.arange(32, dtype=torch.int32, device="cuda").repeat(cfg.n_kv_heads, 1).contiguous()
    L.dom_fc_host = L.dom_fc.cpu().numpy()
    dims = dims_for(cfg)
    kd = build_kdom(L, dims)
    out = torch.empty((1, 4, 64), dtype=torch.float32, device="cuda")
    fasa_decode_step(L.q, L.pos, L.k, L.v, kd, L.dom_fc, L.seq_lens, 1024, out, dims=dims)
    q_rot = torch.empty((1, 4, 64), dtype=torch.float32, device="cuda")
    fasa_apply_rope_q(L.q, L.pos, q_rot, dims)
    sc = torch.empty((1, 2, 1024), dtype=torch.float32, device="cuda")
    fasa_tip_score(q_rot, kd, L.dom_fc, L.seq_lens, sc, dims)
    for h in range(2):
        ref = oracle_unit(L, 0, h, 1024)
        full = ref["K"] @ ref["q_rot"].sum(0)
        P.check_scores(sc[0, h].cpu().numpy(), full)
        dense = O.focused_attention_unit(ref["q_rot"], ref["K"], ref["V"], np.arange(1024))
        P.check_output(out[0, 2 * h:2 * h + 2].cpu().numpy(), dense, "f32")


def test_deterministic():
    """Two runs give bit-identical outputs and indices (no races in the
    cluster reductions)."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_decode_step
    cfg = _cfg("llama3_8b_ctx32k", context=16384, batch=2)
    L = _layer(cfg)
    dims = dims_for(cfg)
    kd = build_kdom(L, dims)
    res = []
    for _ in range(2):
        out = torch.empty((2, 32, 128), dtype=torch.float32, device="cuda")
        idx = torch.empty((2, 8, 256), dtype=torch.int32, device="cuda")
        fasa_decode_step(L.q, L.pos, L.k, L.v, kd, L.dom_fc, L.seq_lens, 256, out, idx, None, None, dims)
        res.append((out.cpu().numpy(), idx.cpu().numpy()))
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])


def test_device_input_checks():
    """Out-of-range device-resident values are clamped and reported in the
    device status word instead of being dereferenced."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_decode_step, fasa_device_status
    cfg = _cfg("tiny_fp32_ctx1k")
    L = _layer(cfg)
    dims = dims_for(cfg)
    kd = build_kdom(L, dims)
    assert fasa_device_status() == 0
    bad_lens = torch.tensor([5000], dtype=torch.int32, device="cuda")
    out = torch.empty((1, 4, 64), dtype=torch.float32, device="cuda")
    fasa_decode_step(L.q, L.pos, L.k, L.v, kd, L.dom_fc, bad_lens, 64, out, dims=dims)
    assert fasa_device_status() & 1
    assert fasa_device_status() == 0
    assert np.all(np.isfinite(out.cpu().numpy()))
