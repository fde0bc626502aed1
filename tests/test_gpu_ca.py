"""Contextual Agreement and the calibration of the dominant FCs (GPU).

fasa_fc_agreement computes, per (batch, KV head, FC), Eq. 4 of "The
Functional Sparsity Hypothesis and the Contextual Agreement (CA) Metric":
|TopK-I(full) & TopK-I(alpha_i)| / K' in fp32 arithmetic; the oracle does
the same in fp64 on the same rotated queries and stored keys.  The two may
take different tokens only where a score lies within the near-tie band of
its set's K'-th score, so a unit's count of common tokens may differ by at
most the number of such tokens (both sets together).  With integer-valued
inputs every fp32 score is exact and the CA must equal the oracle's exactly,
which also checks the tie rule (equal scores: the smaller token first).
fasa_select_dominant_fcs (Algorithm 1's last step) is a rank over the same
fp32 means and must equal the oracle's choice exactly.
"""

import numpy as np
import pytest

import oracle as O
from tests import parity as P
from tests.gpu_util import ensure_built
from workload import configs, gpu_gen

pytestmark = pytest.mark.gpu

# near-tie band of a TopK-I boundary, relative to max(|K'-th score|, RMS of
# the scores): fp32 sums of at most 2 x 64 products of exact inputs are off by
# ~1e-6 of that scale
BAND_RTOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    ensure_built()


def _band(s, kk):
    if kk == 0 or kk >= len(s):
        return 0
    kth = np.sort(s)[::-1][kk - 1]
    tol = BAND_RTOL * max(abs(kth), np.sqrt(np.mean(s ** 2)))
    return int(np.count_nonzero(np.abs(s - kth) <= tol)) - 1


def _gpu_ca(q_rot, k, lens, K, dims):
    import torch
    from kv_cache_token_tip_gb300 import fasa_device_status, fasa_fc_agreement
    ca = torch.full((dims.batch, dims.n_kv_heads, dims.head_dim // 2), float("nan"), dtype=torch.float32,
                    device="cuda")
    fasa_fc_agreement(q_rot, k, lens, K, ca, dims)
    assert fasa_device_status() == 0
    return ca


def _check_unit(ca_gpu, q_rot_g, K_rows, K, exact=False):
    """ca_gpu [d/2] of one (batch, KV head) against the oracle."""
    t = K_rows.shape[0]
    kk = min(K, t)
    if kk == 0:   # both sets empty: Eq. 4 read as full agreement, as the oracle's ca_from_scores
        assert np.all(ca_gpu == 1.0)
        return 0
    ref = O.contextual_agreement_unit(q_rot_g, K_rows, K)
    n_gpu = np.round(np.asarray(ca_gpu, dtype=np.float64) * kk)
    # the value is the fp32 quotient of a count by K'
    assert np.array_equal(np.float32(n_gpu) / np.float32(kk), np.asarray(ca_gpu, dtype=np.float32)), \
        "CA is not a count over K'"
    if exact:
        assert np.array_equal(n_gpu, np.round(ref * kk))
        return 0
    A = O.fc_scores_unit(q_rot_g, K_rows)
    full = A.sum(axis=0)
    bf = _band(full, kk)
    worst = 0
    for i in range(A.shape[0]):
        d = abs(int(n_gpu[i]) - int(round(ref[i] * kk)))
        assert d <= bf + _band(A[i], kk), f"FC {i}: {d} tokens apart beyond the near-tie band"
        worst = max(worst, d)
    return worst


CASES = [
    # (config, overrides, lengths, K)
    ("llama3_8b_ctx32k", dict(context=8192, batch=3), [5001, 8192, 0], 256),   # ragged tails
    ("qwen25_7b_b8_ctx16k", dict(context=4096, batch=2), [4096, 701], 1000),
    ("llama3_8b_ctx32k", dict(context=1024, batch=2), [100, 1000], 256),   # t < K: CA = 1
    ("tiny_fp32_ctx1k", dict(batch=2), [1024, 5], 64),
]


@pytest.mark.parametrize("name,over,lens,K", CASES, ids=[f"{c[0]}-{c[2][0]}" for c in CASES])
def test_fc_agreement_against_oracle(name, over, lens, K):
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_apply_rope_q
    cfg = configs.CONFIGS[name].with_(**over)
    L = gpu_gen.make_layer(cfg, 0)
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    dims = dims_for(cfg)
    q_rot = torch.empty((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32, device="cuda")
    fasa_apply_rope_q(L.q, lens_d, q_rot, dims)
    ca = _gpu_ca(q_rot, L.k, lens_d, K, dims).cpu().numpy()
    qr = q_rot.cpu().numpy().astype(np.float64)
    G = cfg.group
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            K_rows = P.host_f64(L.k[b, h, :lens[b]], cfg.dtype)
            _check_unit(ca[b, h], qr[b, h * G:(h + 1) * G], K_rows, K)
            if lens[b] <= K:
                assert np.all(ca[b, h] == 1.0)


def test_fc_agreement_exact_on_integer_inputs():
    """Integer keys and queries: every fp32 score is exact, scores tie often,
    and the GPU's CA equals the oracle's exactly."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for
    cfg = configs.CONFIGS["llama3_8b_ctx32k"].with_(context=2048, batch=2, n_q_heads=8, n_kv_heads=2)
    rng = np.random.default_rng(21)
    B, Hq, H, T, d = cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.context, cfg.head_dim
    k = rng.integers(-4, 5, size=(B, H, T, d)).astype(np.float32)
    q = rng.integers(-3, 4, size=(B, Hq, d)).astype(np.float32)
    k_d = torch.from_numpy(k).cuda().to(torch.bfloat16)
    q_d = torch.from_numpy(q).cuda()
    lens = [2048, 1500]
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    dims = dims_for(cfg)
    for K in (100, 1024):
        ca = _gpu_ca(q_d, k_d, lens_d, K, dims).cpu().numpy()
        G = Hq // H
        for b in range(B):
            for h in range(H):
                _check_unit(ca[b, h], q[b, h * G:(h + 1) * G].astype(np.float64),
                            k[b, h, :lens[b]].astype(np.float64), K, exact=True)


@pytest.mark.parametrize("case", ["large_k", "sample_misses"])
def test_fc_agreement_threshold_fallbacks(case):
    """The threshold search falls back to a select over whole rows when the
    candidate list overflows (a large K') or holds fewer than K' keys (every
    16th token scores far above the rest, so the sample overestimates the
    K'-th score).  Integer inputs: the result equals the oracle's exactly."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for
    cfg = configs.CONFIGS["llama3_8b_ctx32k"].with_(context=8192, batch=1, n_q_heads=4, n_kv_heads=1)
    rng = np.random.default_rng(5)
    T, d = cfg.context, cfg.head_dim
    if case == "large_k":
        k = rng.integers(-4, 5, size=(1, 1, T, d)).astype(np.float32)
        q = rng.integers(-3, 4, size=(1, 4, d)).astype(np.float32)
        K = 3000
    else:
        k = rng.integers(-1, 2, size=(1, 1, T, d)).astype(np.float32)
        k[0, 0, ::16] = 4.0
        q = np.ones((1, 4, d), dtype=np.float32)
        K = 2000
    k_d = torch.from_numpy(k).cuda().to(torch.bfloat16)
    lens_d = torch.tensor([T], dtype=torch.int32, device="cuda")
    ca = _gpu_ca(torch.from_numpy(q).cuda(), k_d, lens_d, K, dims_for(cfg)).cpu().numpy()
    _check_unit(ca[0, 0], q[0].astype(np.float64), k[0, 0].astype(np.float64), K, exact=True)


def _gpu_cca(q_rot, k, dom, lens, K, dims):
    import torch
    from kv_cache_token_tip_gb300 import fasa_compound_agreement, fasa_device_status
    cca = torch.full((dims.batch, dims.n_kv_heads), float("nan"), dtype=torch.float32, device="cuda")
    fasa_compound_agreement(q_rot, k, dom, lens, K, cca, dims)
    assert fasa_device_status() == 0
    return cca.cpu().numpy()


def test_compound_agreement_against_oracle():
    """Compound CA of the layer's dominant sets against the oracle (near-tie
    band on both boundaries), plus two identities that must hold bit for bit:
    the set of every FC gives 1, and a one-FC set gives that FC's CA."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_apply_rope_q
    cfg = configs.CONFIGS["llama3_8b_ctx32k"].with_(context=8192, batch=3)
    L = gpu_gen.make_layer(cfg, 0)
    lens = [8192, 3003, 0]
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    dims = dims_for(cfg)
    q_rot = torch.empty((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32, device="cuda")
    fasa_apply_rope_q(L.q, lens_d, q_rot, dims)
    K = cfg.budget
    cca = _gpu_cca(q_rot, L.k, L.dom_fc, lens_d, K, dims)
    qr = q_rot.cpu().numpy().astype(np.float64)
    G = cfg.group
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            if lens[b] == 0:
                assert cca[b, h] == 1.0
                continue
            q_g = qr[b, h * G:(h + 1) * G]
            K_rows = P.host_f64(L.k[b, h, :lens[b]], cfg.dtype)
            dom = L.dom_fc_host[h]
            ref = O.compound_agreement_unit(q_g, K_rows, dom, K)
            A = O.fc_scores_unit(q_g, K_rows)
            kk = min(K, lens[b])
            band = _band(A.sum(axis=0), kk) + _band(A[dom].sum(axis=0), kk)
            assert abs(round(cca[b, h] * kk) - round(ref * kk)) <= band
    # every FC: the summed scores are the full scores
    all_fc = torch.arange(cfg.head_dim // 2, dtype=torch.int32, device="cuda").repeat(cfg.n_kv_heads, 1)
    d_all = dims_for(cfg, n_tip=cfg.head_dim // 2)
    assert np.all(_gpu_cca(q_rot, L.k, all_fc.contiguous(), lens_d, K, d_all) == 1.0)
    # one FC per head: equals fasa_fc_agreement's value for that FC
    ca = _gpu_ca(q_rot, L.k, lens_d, K, dims).cpu().numpy()
    for i in (0, 17, 63):
        one = torch.full((cfg.n_kv_heads, 1), i, dtype=torch.int32, device="cuda")
        got = _gpu_cca(q_rot, L.k, one, lens_d, K, dims_for(cfg, n_tip=1))
        assert np.array_equal(got, ca[:, :, i])


def test_compound_agreement_fp32_and_ragged_sets():
    """fp32 keys, 64-dim heads, and dominant rows that end early (-1): the
    compound CA reads each head's set as the entries before its first -1."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_apply_rope_q
    cfg = configs.CONFIGS["tiny_fp32_ctx1k"].with_(batch=2)
    L = gpu_gen.make_layer(cfg, 0)
    lens = [1024, 300]
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    dom = np.array([[3, 9, 17, -1, -1, -1], [0, 1, 2, 3, 30, 31]], dtype=np.int32)
    dims = dims_for(cfg, n_tip=dom.shape[1])
    q_rot = torch.empty((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32, device="cuda")
    fasa_apply_rope_q(L.q, lens_d, q_rot, dims)
    K = 64
    cca = _gpu_cca(q_rot, L.k, torch.from_numpy(dom).cuda(), lens_d, K, dims)
    qr = q_rot.cpu().numpy().astype(np.float64)
    G = cfg.group
    for b in range(cfg.batch):
        for h in range(cfg.n_kv_heads):
            q_g = qr[b, h * G:(h + 1) * G]
            K_rows = P.host_f64(L.k[b, h, :lens[b]], cfg.dtype)
            ref = O.compound_agreement_unit(q_g, K_rows, dom[h], K)
            A = O.fc_scores_unit(q_g, K_rows)
            kk = min(K, lens[b])
            band = _band(A.sum(axis=0), kk) + _band(A[O.dominant_set(dom[h])].sum(axis=0), kk)
            assert abs(round(cca[b, h] * kk) - round(ref * kk)) <= band


def test_select_dominant_equals_oracle_with_ties():
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_select_dominant_fcs
    cfg = configs.CONFIGS["llama3_8b_ctx32k"]
    dims = dims_for(cfg)
    rng = np.random.default_rng(4)
    # means on a coarse grid: many equal values, ordered by FC index
    ca_mean = (rng.integers(0, 9, size=(cfg.n_kv_heads, cfg.head_dim // 2)) / 8.0).astype(np.float32)
    for n in (1, 8, 16, 63, 64):
        dom = torch.full((cfg.n_kv_heads, n), -1, dtype=torch.int32, device="cuda")
        fasa_select_dominant_fcs(torch.from_numpy(ca_mean).cuda(), n, dom, dims)
        assert np.array_equal(dom.cpu().numpy(), O.calibrate_dominant_fcs(ca_mean.astype(np.float64), n))


def test_calibration_pipeline_recovers_the_outlier_fcs():
    """CA over a batch of synthetic sequences, averaged, then the n_tip FCs of
    highest mean CA.  The choice equals the oracle's on the same means, and the
    FCs the generator made dominant (large-magnitude outlier FCs that carry the
    logits) are among those chosen."""
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_apply_rope_q, fasa_select_dominant_fcs
    from workload import synth
    cfg = configs.CONFIGS["llama3_8b_ctx32k"].with_(context=4096, batch=4)
    L = gpu_gen.make_layer(cfg, 0)
    lens_d = torch.full((cfg.batch,), cfg.context, dtype=torch.int32, device="cuda")
    dims = dims_for(cfg)
    q_rot = torch.empty((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32, device="cuda")
    fasa_apply_rope_q(L.q, lens_d, q_rot, dims)
    ca = _gpu_ca(q_rot, L.k, lens_d, cfg.budget, dims)
    ca_mean = ca.mean(dim=0).contiguous()
    dom = torch.empty((cfg.n_kv_heads, cfg.n_tip), dtype=torch.int32, device="cuda")
    fasa_select_dominant_fcs(ca_mean, cfg.n_tip, dom, dims)
    got = dom.cpu().numpy()
    assert np.array_equal(got, O.calibrate_dominant_fcs(ca_mean.cpu().numpy().astype(np.float64), cfg.n_tip))
    # the planted outlier FCs are the n_outlier FCs of highest mean CA (the
    # fp64 oracle on the same recipe shows a gap of >= 0.06 below them)
    outl = synth.outlier_fcs(cfg, 0)
    m = ca_mean.cpu().numpy()
    for h in range(cfg.n_kv_heads):
        top = np.argsort(-m[h], kind="stable")[:cfg.n_outlier]
        assert set(top.tolist()) == set(outl[h].tolist())
        assert set(outl[h].tolist()) <= set(got[h].tolist())


def test_fc_agreement_rejects_bad_arguments():
    import torch
    from kv_cache_token_tip_gb300 import FasaError, dims_for, fasa_device_status, fasa_fc_agreement, \
        fasa_select_dominant_fcs
    cfg = configs.CONFIGS["llama3_8b_ctx32k"].with_(context=1024, batch=1)
    L = gpu_gen.make_layer(cfg, 0)
    q_rot = torch.zeros((1, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32, device="cuda")
    ca = torch.empty((1, cfg.n_kv_heads, cfg.head_dim // 2), dtype=torch.float32, device="cuda")
    with pytest.raises(FasaError) as e:
        fasa_fc_agreement(q_rot, L.k, L.seq_lens, 0, ca, dims_for(cfg))
    assert e.value.status == 1
    # a workspace smaller than the size query asks for
    from kv_cache_token_tip_gb300 import fasa_fc_agreement_workspace_size
    n = fasa_fc_agreement_workspace_size(dims_for(cfg))
    assert n == cfg.batch * cfg.n_kv_heads * (cfg.head_dim // 2 + 1) * (cfg.context + cfg.context // 32) * 4
    short = torch.empty(n - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(FasaError) as e:
        fasa_fc_agreement(q_rot, L.k, L.seq_lens, 64, ca, dims_for(cfg), workspace=short)
    assert e.value.status == 3
    dom = torch.empty((cfg.n_kv_heads, 65), dtype=torch.int32, device="cuda")
    with pytest.raises(FasaError) as e:
        fasa_select_dominant_fcs(ca[0], 65, dom, dims_for(cfg))
    assert e.value.status == 1
    # an out-of-range length is clamped and reported on the device
    assert fasa_device_status() == 0
    bad = torch.tensor([5000], dtype=torch.int32, device="cuda")
    fasa_fc_agreement(q_rot, L.k, bad, 64, ca, dims_for(cfg))
    assert fasa_device_status() & 1
    assert np.all(np.isfinite(ca.cpu().numpy()))
