"""C-ABI surface and host-side logic, without a GPU: the library loads, exports
every symbol the header declares, and rejects bad arguments before touching
CUDA.  Also the byte model and the synthetic generator."""

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fasa.h")


@pytest.fixture(scope="module")
def L():
    from kv_cache_token_tip_gb300 import build, lib
    build.build()
    return lib()


def header_symbols():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fasa_[a-z_]+)\s*\(", src)))


def test_header_declares_the_decode_path_calls():
    syms = header_symbols()
    for name in ("fasa_apply_rope_q", "fasa_tip_score", "fasa_topk_select", "fasa_focused_attention",
                 "fasa_decode_step", "fasa_dense_attention", "fasa_build_kdom", "fasa_append_kdom",
                 "fasa_workspace_size", "fasa_device_status", "fasa_decode_step_append",
                 "fasa_decode_step_split", "fasa_decode_step_append_split", "fasa_build_knondom",
                 "fasa_fc_agreement", "fasa_compound_agreement", "fasa_select_dominant_fcs"):
        assert name in syms


def test_every_declared_symbol_is_exported(L):
    for name in header_symbols():
        assert hasattr(L, name), f"{name} not exported"
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_binding_covers_every_symbol():
    from kv_cache_token_tip_gb300 import fasa
    assert sorted(fasa.EXPORTS) == header_symbols()


def _dims(**kw):
    from kv_cache_token_tip_gb300 import FasaDims
    d = dict(batch=1, n_q_heads=32, n_kv_heads=8, head_dim=128, t_max=32768, n_tip=16, dtype=1,
             reserved=0, rope_theta=5e5)
    d.update(kw)
    return FasaDims(d["batch"], d["n_q_heads"], d["n_kv_heads"], d["head_dim"], d["t_max"], d["n_tip"],
                    d["dtype"], d["reserved"], d["rope_theta"])


BAD_DIMS = [
    (dict(batch=0), 1), (dict(n_q_heads=30), 1), (dict(t_max=1000), 1), (dict(n_tip=0), 1),
    (dict(n_tip=65), 1), (dict(rope_theta=0.0), 1), (dict(rope_theta=float("inf")), 1),
    (dict(reserved=17), 1), (dict(reserved=-1), 1), (dict(head_dim=96), 2), (dict(head_dim=7), 1),
    (dict(dtype=5), 2), (dict(n_q_heads=72, n_kv_heads=8), 2),
]


@pytest.mark.parametrize("kw,code", BAD_DIMS)
def test_bad_dims_rejected_before_launch(L, kw, code):
    d = _dims(**kw)
    P = 0x10000  # never dereferenced: validation fails first
    st = L.fasa_decode_step(P, P, P, P, P, P, P, 256, P, None, None, None, 0, ctypes.byref(d), None)
    assert st == code
    assert L.fasa_tip_score(P, P, P, P, P, ctypes.byref(d), None) == code
    assert L.fasa_apply_rope_q(P, P, P, ctypes.byref(d), None) == code
    assert L.fasa_dense_attention(P, P, P, P, P, ctypes.byref(d), None) == code


def test_null_and_misaligned_pointers_rejected(L):
    d = _dims()
    P = 0x10000
    assert L.fasa_decode_step(None, P, P, P, P, P, P, 256, P, None, None, None, 0, ctypes.byref(d), None) == 1
    assert L.fasa_decode_step(P, P, P + 8, P, P, P, P, 256, P, None, None, None, 0, ctypes.byref(d), None) == 1
    assert L.fasa_decode_step(P, P, P, P, P, P, P, 0, P, None, None, None, 0, ctypes.byref(d), None) == 1
    assert L.fasa_decode_step(P, P, P, P, P, P, P, 256, P, None, None, None, 0, None, None) == 1
    assert L.fasa_topk_select(P, P, 0, P, P, ctypes.byref(d), None) == 1
    assert L.fasa_topk_select(P + 4, P, 10, P, P, ctypes.byref(d), None) == 1
    assert L.fasa_focused_attention(P, P, P, P, P, None, 10, P, ctypes.byref(d), None) == 1
    assert L.fasa_build_kdom(P, P, None, P + 2, ctypes.byref(d), None) == 1
    assert L.fasa_append_kdom(P, None, P, P, ctypes.byref(d), None) == 1
    assert L.fasa_device_status(None, None) == 1


def test_split_step_arguments_rejected_before_launch(L):
    """FASA-M split keys: bf16 and N_tip a multiple of 4 only (the K^nondom
    row must be whole 16-byte chunks), checked on the host."""
    P = 0x10000  # never dereferenced: validation fails first
    sp = L.fasa_decode_step_split
    assert sp(P, P, P, P, P, P, P, 256, P, None, None, None, 0, ctypes.byref(_dims(n_tip=6)), None) == 2
    assert sp(P, P, P, P, P, P, P, 256, P, None, None, None, 0, ctypes.byref(_dims(dtype=0)), None) == 2
    assert sp(None, P, P, P, P, P, P, 256, P, None, None, None, 0, ctypes.byref(_dims()), None) == 1
    assert sp(P, P, P + 8, P, P, P, P, 256, P, None, None, None, 0, ctypes.byref(_dims()), None) == 1
    ap = L.fasa_decode_step_append_split
    assert ap(P, P, P, P, P, P, P, P, 256, P, None, None, None, 0, ctypes.byref(_dims(n_tip=6)), None) == 2
    assert ap(P, P, P, P, P, P, P, P, 256, P, None, None, None, 0, ctypes.byref(_dims(dtype=0)), None) == 2
    assert ap(P, P, P, P, P + 8, P, P, P, 256, P, None, None, None, 0, ctypes.byref(_dims()), None) == 1
    assert ap(P, None, P, P, P, P, P, P, 256, P, None, None, None, 0, ctypes.byref(_dims()), None) == 1
    assert L.fasa_build_knondom(P, P, None, P + 2, ctypes.byref(_dims()), None) == 1
    assert L.fasa_build_knondom(P, None, None, P, ctypes.byref(_dims()), None) == 1


def test_calibration_arguments_rejected_before_launch(L):
    """The calibration entry points validate on the host: dims, null and
    misaligned pointers, K < 1, n_tip outside 1..d/2, a missing or short
    workspace -- all before any CUDA call."""
    d = _dims()
    P = 0x10000
    need = ctypes.c_size_t(0)
    assert L.fasa_fc_agreement_workspace_size(ctypes.byref(d), ctypes.byref(need)) == 0
    units, F, T = d.batch * d.n_kv_heads, d.head_dim // 2, d.t_max
    assert need.value == units * (F + 1) * (T + T // 32) * 4
    ws, n = P, need.value
    assert L.fasa_fc_agreement_workspace_size(ctypes.byref(d), None) == 1
    bad = _dims(n_tip=0)
    assert L.fasa_fc_agreement_workspace_size(ctypes.byref(bad), ctypes.byref(need)) == 1
    assert need.value == 0
    fa = L.fasa_fc_agreement
    assert fa(P, P, P, 256, P, ws, n, ctypes.byref(bad), None) == 1
    assert fa(None, P, P, 256, P, ws, n, ctypes.byref(d), None) == 1
    assert fa(P, P + 8, P, 256, P, ws, n, ctypes.byref(d), None) == 1    # k_cache not 16-byte aligned
    assert fa(P, P, P, 0, P, ws, n, ctypes.byref(d), None) == 1
    assert fa(P, P, P, 256, P, None, n, ctypes.byref(d), None) == 3
    assert fa(P, P, P, 256, P, ws, n - 1, ctypes.byref(d), None) == 3
    assert fa(P, P, P, 256, P, ws + 4, n, ctypes.byref(d), None) == 3  # workspace not 16-byte aligned
    ca = L.fasa_compound_agreement
    assert ca(P, P, None, P, 256, P, ws, n, ctypes.byref(d), None) == 1
    assert ca(P, P, P, P, 0, P, ws, n, ctypes.byref(d), None) == 1
    assert ca(P, P, P, P, 256, P, ws, n - 16, ctypes.byref(d), None) == 3
    sd = L.fasa_select_dominant_fcs
    assert sd(P, 0, P, ctypes.byref(d), None) == 1
    assert sd(P, F + 1, P, ctypes.byref(d), None) == 1
    assert sd(None, 4, P, ctypes.byref(d), None) == 1
    assert sd(P, 4, None, ctypes.byref(d), None) == 1


def test_status_strings(L):
    for code, name in ((0, b"FASA_OK"), (1, b"FASA_ERR_INVALID_ARG"), (2, b"FASA_ERR_UNSUPPORTED"),
                       (3, b"FASA_ERR_WORKSPACE"), (4, b"FASA_ERR_CUDA"), (99, b"FASA_ERR_UNKNOWN")):
        assert L.fasa_status_string(code) == name


def test_byte_model_matches_pages_fraction():
    """The bench's byte count divided by a dense K+V read is the pages'
    fraction N_tip/d + N_fac/t (plus the query/output terms)."""
    import bench
    import oracle as O
    from workload import configs
    for name in ("llama3_8b_ctx32k", "qwen25_7b_b8_ctx16k", "llama3_8b_b4_ctx128k"):
        cfg = configs.CONFIGS[name]
        lens = np.full(cfg.batch, cfg.context)
        m = bench.algorithmic_bytes(cfg, lens)
        dense_kv = cfg.batch * cfg.n_kv_heads * cfg.context * 2 * cfg.head_dim * cfg.elem_bytes
        frac = (m["tip"] + m["fac"]) / dense_kv
        assert np.isclose(frac, O.bytes_fraction(cfg.n_tip, cfg.head_dim, cfg.budget, cfg.context), rtol=1e-12)
    cfg = configs.CONFIGS["llama3_8b_ctx32k"]
    assert abs(bench.algorithmic_bytes(cfg, [32768])["total"] / 1e6 - 17.85) < 0.01


def test_generator_deterministic_and_recipe():
    from workload import configs, synth
    cfg = configs.CONFIGS["tiny_fp32_ctx1k"].with_(context=64)
    a = synth.gen_layer(cfg, 0)
    b = synth.gen_layer(cfg, 0)
    assert np.array_equal(a.k, b.k) and np.array_equal(a.q, b.q)
    c = synth.gen_layer(cfg, 1)
    assert not np.array_equal(a.k, c.k)
    # outlier FCs are in the dominant table and carry ~8x the energy
    dom = synth.dominant_fcs(cfg, 0)
    outl = synth.outlier_fcs(cfg, 0)
    for h in range(cfg.n_kv_heads):
        assert set(outl[h]) <= set(dom[h]) and len(set(dom[h])) == cfg.n_tip
    k, _ = synth.gen_kv_head(cfg.with_(context=4096), 0, 0, 0)
    e = (k[:, 0::2] ** 2 + k[:, 1::2] ** 2).mean(0)
    assert np.all(e[outl[0]] > 30) and np.median(e) < 3
    # bf16 rounding is nearest-even
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5], dtype=np.float32)
    assert list(synth.f32_to_bf16_bits(x)) == [0x3F80, 0x3F80, 0x3F82, 0xC020]


def test_ragged_lengths_in_range():
    from workload import configs, synth
    cfg = configs.CONFIGS["mistral_7b_l32_b32_ragged"]
    lens = synth.seq_lens(cfg)
    assert lens.shape == (32,) and lens.min() >= 4096 and lens.max() <= 32768


def test_fasa_m_memory_model_is_eq10():
    """bench.py's FASA-M footprint estimate is Eq. 10 of the oracle, summed
    over the (batch, KV head) units of one layer."""
    import bench
    import oracle as O
    from workload import configs
    for name in ("llama3_8b_ctx32k", "qwen25_7b_b8_ctx16k", "llama3_8b_b4_ctx128k", "tiny_fp32_ctx1k"):
        cfg = configs.CONFIGS[name]
        ref = cfg.batch * cfg.n_kv_heads * O.fasa_m_gpu_bytes(1, cfg.context, cfg.head_dim, cfg.n_tip, cfg.budget,
                                                               cfg.elem_bytes)
        assert bench.fasa_m_eq10_bytes(cfg) == ref


def test_variant_workloads():
    """The per-head, all-FC and pyramid-budget workloads: each head's row holds
    its own count of distinct FCs (its outlier FCs first in the draw) padded
    with -1; every FC is dominant in the all-FC workload; the pyramid budgets
    fall from 384 to 128 with mean 256 and the byte model follows them."""
    import bench
    import oracle as O
    from workload import configs, synth
    cfg = configs.CONFIGS["llama3_8b_ctx32k_ragged_ntip"]
    dom = synth.dominant_fcs(cfg, 0)
    outl = synth.outlier_fcs(cfg, 0)
    assert dom.shape == (cfg.n_kv_heads, cfg.n_tip) and cfg.n_tip == max(cfg.n_tip_per_head)
    for h in range(cfg.n_kv_heads):
        s = O.dominant_set(dom[h])
        assert len(s) == cfg.n_tip_per_head[h] == len(set(s))
        assert all(0 <= i < cfg.n_fc for i in s) and np.all(dom[h, len(s):] == -1)
        assert set(outl[h][:min(cfg.n_outlier, len(s))].tolist()) <= set(s)
    assert sum(cfg.n_tip_per_head) == 16 * cfg.n_kv_heads
    ok = configs.CONFIGS["llama3_8b_ctx32k_oraclek"]
    assert np.array_equal(synth.dominant_fcs(ok, 0), np.tile(np.arange(ok.n_fc), (ok.n_kv_heads, 1)))
    py = configs.CONFIGS["mistral_7b_l32_b32_pyramid"]
    b = py.budget_per_layer
    assert len(b) == py.layers and b[0] == 384 and b[-1] == 128 and sum(b) == 256 * py.layers
    assert all(x >= y for x, y in zip(b, b[1:])) and max(b) == py.budget
    lens = synth.seq_lens(py)
    uni = configs.CONFIGS["mistral_7b_l32_b32_ragged"]
    tot_py = sum(bench.algorithmic_bytes(py, lens, py.layer_budget(l))["fac"] for l in range(py.layers))
    tot_uni = bench.algorithmic_bytes(uni, lens)["fac"] * uni.layers
    assert abs(tot_py - tot_uni) < 0.01 * tot_uni   # same mean budget, lengths mostly above 384


def test_fault_injection_arguments_validated(L):
    """The test hook rejects a zero wait bound and indices below -1, and
    accepts (then restores) the defaults; it only sets host-side values."""
    f = L.fasa_test_fault_injection
    assert f(0, -1, -1) == 1
    assert f(1000000000, -2, -1) == 1
    assert f(1000000000, -1, -2) == 1
    assert f(2000000, 0, 3) == 0
    assert f(1000000000, -1, -1) == 0
