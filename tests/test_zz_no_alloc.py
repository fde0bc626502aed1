"""fasa_decode_step_noalloc, the entry point for callers that cannot allocate
device memory (for example a plug-in whose host owns every device allocation,
or a service that forbids allocations once it serves).  It must give the same
result as fasa_decode_step with a caller-provided workspace.  This file runs
last so that a failure here never hides the other tests."""

import numpy as np
import pytest

from tests.gpu_util import build_kdom, ensure_built
from workload import configs, gpu_gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    ensure_built()


def _dims():
    from kv_cache_token_tip_gb300 import dims_for
    # two CTAs per unit: each holds 16K tokens, more than shared memory keeps,
    # so the step needs its score workspace
    return dims_for(configs.CONFIGS["llama3_8b_ctx32k"], cluster_ctas=2)


def test_noalloc_matches_workspace_entry_point_twice():
    import torch
    from kv_cache_token_tip_gb300 import fasa_decode_step, fasa_decode_step_noalloc, fasa_device_status, \
        fasa_workspace_size
    from tests import parity as P
    cfg = configs.CONFIGS["llama3_8b_ctx32k"]
    dims = _dims()
    ws_bytes = fasa_workspace_size(dims, cfg.budget)
    assert 0 < ws_bytes <= (16 << 20)
    for layer in (0, 1):   # two calls in a row, different inputs
        L = gpu_gen.make_layer(cfg, layer)
        kd = build_kdom(L, dims)
        shape_o = (cfg.batch, cfg.n_q_heads, cfg.head_dim)
        shape_i = (cfg.batch, cfg.n_kv_heads, cfg.budget)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        out_ref = torch.empty(shape_o, dtype=torch.float32, device="cuda")
        idx_ref = torch.empty(shape_i, dtype=torch.int32, device="cuda")
        fasa_decode_step(L.q, L.pos, L.k, L.v, kd, L.dom_fc, L.seq_lens, cfg.budget, out_ref, idx_ref, None,
                         ws, dims)
        out = torch.full(shape_o, float("nan"), dtype=torch.float32, device="cuda")
        idx = torch.empty(shape_i, dtype=torch.int32, device="cuda")
        cnt = torch.empty((cfg.batch, cfg.n_kv_heads), dtype=torch.int32, device="cuda")
        fasa_decode_step_noalloc(L.q, L.pos, L.k, L.v, kd, L.dom_fc, L.seq_lens, cfg.budget, out, idx, cnt,
                                 dims)
        assert fasa_device_status() == 0
        assert np.array_equal(idx.cpu().numpy(), idx_ref.cpu().numpy())
        assert np.all(cnt.cpu().numpy() == cfg.budget)
        P.check_output(out.cpu().numpy(), out_ref.cpu().numpy(), "bf16")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import ctypes
    from kv_cache_token_tip_gb300 import dims_for, fasa_workspace_size, lib
    cfg = configs.CONFIGS["llama3_8b_b4_ctx128k"].with_(batch=5)   # 5*8*131072*4 B = 20 MiB > 16 MiB
    dims = dims_for(cfg, cluster_ctas=4)
    # the size check must come first: with the plan's workspace beyond the
    # scratch, the call returns before it looks at (or launches on) any
    # pointer, so null pointers are safe here
    assert fasa_workspace_size(dims, cfg.budget) > (16 << 20)
    st = lib().fasa_decode_step_noalloc(None, None, None, None, None, None, None, cfg.budget, None, None, None,
                                        ctypes.byref(dims), None)
    assert st == 3   # FASA_ERR_WORKSPACE, before any launch


def test_noalloc_falls_back_to_a_cluster_size_that_fits():
    """One layer of the 32-sequence ragged batch: the automatic plan (one CTA
    per unit, 32K-token ranges) needs a 32 MiB score workspace, more than the
    scratch; the no-alloc entry point runs a larger cluster instead, with the
    result of the workspace entry point forced to that cluster size."""
    import torch
    from kv_cache_token_tip_gb300 import (dims_for, fasa_cluster_size, fasa_decode_step, fasa_decode_step_noalloc,
                                          fasa_device_status, fasa_workspace_size)
    cfg = configs.CONFIGS["mistral_7b_l32_b32_ragged"]
    auto = dims_for(cfg)
    assert fasa_workspace_size(auto, cfg.budget) > (16 << 20)
    sizes = [c for c in (2, 4, 8, 16) if fasa_workspace_size(dims_for(cfg, cluster_ctas=c), cfg.budget) <= (16 << 20)]
    assert sizes
    forced = dims_for(cfg, cluster_ctas=sizes[0])
    assert fasa_cluster_size(forced) == sizes[0]
    L = gpu_gen.make_layer(cfg, 0)
    kd = build_kdom(L, forced)
    shape_o = (cfg.batch, cfg.n_q_heads, cfg.head_dim)
    ws_bytes = fasa_workspace_size(forced, cfg.budget)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda") if ws_bytes else None
    out_ref = torch.empty(shape_o, dtype=torch.float32, device="cuda")
    fasa_decode_step(L.q, L.pos, L.k, L.v, kd, L.dom_fc, L.seq_lens, cfg.budget, out_ref, None, None, ws, forced)
    out = torch.full(shape_o, float("nan"), dtype=torch.float32, device="cuda")
    fasa_decode_step_noalloc(L.q, L.pos, L.k, L.v, kd, L.dom_fc, L.seq_lens, cfg.budget, out, None, None, auto)
    assert fasa_device_status() == 0
    assert np.array_equal(out.cpu().numpy(), out_ref.cpu().numpy())
