"""Shared helpers of the GPU parity tests (library vs oracle on the same bytes)."""

import numpy as np

import oracle as O
from tests.parity import host_f64


def ensure_built():
    from kv_cache_token_tip_gb300 import build
    build.build()


def oracle_unit(layer, b, h, budget, n_tip=None):
    """Oracle pass of one (batch, KV head) on the stored device inputs."""
    cfg = layer.cfg
    G = cfg.group
    L = int(layer.seq_lens_host[b])
    q = host_f64(layer.q[b, h * G:(h + 1) * G], cfg.dtype)
    K = host_f64(layer.k[b, h, :L], cfg.dtype)
    V = host_f64(layer.v[b, h, :L], cfg.dtype)
    q_rot = O.apply_rope_q(q[None], np.array([layer.pos_host[b]]), cfg.rope_theta)[0]
    dom = O.dominant_set(layer.dom_fc_host[h])
    s = O.tip_scores_unit(q_rot, K, dom)
    idx = O.topk_select_unit(s, budget)
    out = O.focused_attention_unit(q_rot, K, V, idx)
    return dict(q_rot=q_rot, K=K, V=V, scores=s, idx=idx, out=out)


def build_kdom(layer, dims):
    import torch
    from kv_cache_token_tip_gb300 import fasa_build_kdom
    cfg = layer.cfg
    kd = torch.empty((cfg.batch, cfg.n_kv_heads, cfg.context // 64, dims.n_tip, 64, 2),
                     dtype=layer.k.dtype, device=layer.k.device)
    fasa_build_kdom(layer.k, layer.dom_fc, None, kd, dims)
    return kd
