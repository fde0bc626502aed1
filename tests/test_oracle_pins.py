"""The oracle against its pins (CPU only), and planted mistakes that the pins
must catch."""

import importlib.util
import os

import numpy as np
import pytest

import oracle.fasa_oracle as O
from tests import oracle_pins as P

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "fasa_oracle.py")


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check(O)


def _fresh_oracle():
    spec = importlib.util.spec_from_file_location("oracle_mutant", ORACLE_SRC)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _rope_row_convention(x, pos, rope_theta):
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    th = np.power(float(rope_theta), -2.0 * np.arange(d // 2) / d)
    a = np.asarray(pos, dtype=np.float64)[..., None] * th
    c, s = np.cos(a), np.sin(a)
    y = np.empty_like(x)
    y[..., 0::2] = x[..., 0::2] * c + x[..., 1::2] * s
    y[..., 1::2] = -x[..., 0::2] * s + x[..., 1::2] * c
    return y


def _rope_rotate_half(x, pos, rope_theta):
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    th = np.power(float(rope_theta), -2.0 * np.arange(d // 2) / d)
    a = np.asarray(pos, dtype=np.float64)[..., None] * th
    c, s = np.cos(a), np.sin(a)
    y = np.empty_like(x)
    y[..., :d // 2] = x[..., :d // 2] * c - x[..., d // 2:] * s
    y[..., d // 2:] = x[..., :d // 2] * s + x[..., d // 2:] * c
    return y


def _fc_score_dropped_term(q_vec, k_rows, i):
    return q_vec[2 * i] * k_rows[:, 2 * i]


def _fac_unscaled(q_rot_group, k_rows, v_rows, idx, return_weights=False):
    q = np.atleast_2d(q_rot_group)
    idx = np.asarray(idx, dtype=np.int64)
    out = np.zeros((q.shape[0], q.shape[1]))
    w_all = np.zeros((q.shape[0], idx.shape[0]))
    for g in range(q.shape[0]):
        lg = k_rows[idx] @ q[g]
        w = np.exp(lg - lg.max())
        w /= w.sum()
        w_all[g] = w
        out[g] = w @ v_rows[idx]
    return (out, w_all) if return_weights else out


def _topk_larger_index_first(scores, k):
    s = np.asarray(scores, dtype=np.float64)
    kk = min(int(k), s.shape[0])
    order = np.lexsort((-np.arange(s.shape[0]), -s))
    return np.sort(order[:kk])


def _freq_half_exponent(rope_theta, d):
    return np.power(float(rope_theta), -1.0 * np.arange(d // 2) / d)


def _kdom_wrong_pair(K_stored, dom_fc, block=64):
    B, H, T, _ = K_stored.shape
    n = dom_fc.shape[1]
    out = np.zeros((B, H, T // block, n, block, 2), dtype=K_stored.dtype)
    for h in range(H):
        for j in range(n):
            i = int(dom_fc[h, j])
            if i < 0:
                continue
            out[:, h, :, j] = K_stored[:, h, :, i:i + 2].reshape(B, T // block, block, 2)
    return out


def _focused_attention_wrong_group(q_rot, K, V, idx, count):
    B, Hq, d = q_rot.shape
    Hkv = K.shape[1]
    out = np.zeros((B, Hq, d))
    for b in range(B):
        for hq in range(Hq):
            h = hq % Hkv
            sel = np.asarray(idx[b, h, :int(count[b, h])], dtype=np.int64)
            out[b, hq] = O.focused_attention_unit(q_rot[b, hq:hq + 1], K[b, h], V[b, h], sel)[0]
    return out


def _append_one_position_late(K, V, k_new, v_new, seq_lens, rope_theta):
    K = np.array(K, dtype=np.float64, copy=True)
    V = np.array(V, dtype=np.float64, copy=True)
    lens = np.asarray(seq_lens, dtype=np.int64)
    for b in range(K.shape[0]):
        t = int(lens[b])
        K[b, :, t, :] = O.rope_rotate(np.asarray(k_new[b], dtype=np.float64), t + 1, rope_theta)
        V[b, :, t, :] = np.asarray(v_new[b], dtype=np.float64)
    return K, V, lens + 1


def _ca_over_t(full, alpha_i, K):
    t = len(full)
    kk = min(K, t)
    a = set(O.topk_select_unit(full, kk).tolist())
    b = set(O.topk_select_unit(alpha_i, kk).tolist())
    return len(a & b) / t


def _calibrate_lowest(ca_mean, n_tip):
    return np.sort(np.argsort(np.asarray(ca_mean), axis=1, kind="stable")[:, :n_tip], axis=1).astype(np.int32)


def _ca_fc_vs_itself(q_rot_group, k_rows, K):
    A = O.fc_scores_unit(q_rot_group, k_rows)
    return np.array([O.ca_from_scores(A[i], A[i], K) for i in range(A.shape[0])])


def _compound_drops_last(q_rot_group, k_rows, dom_fc, K):
    if np.asarray(k_rows).shape[0] == 0:
        return 1.0
    A = O.fc_scores_unit(q_rot_group, k_rows)
    dom = list(dom_fc)
    dom = dom[:-1] if len(dom) > 1 else dom
    return O.ca_from_scores(A.sum(axis=0), A[np.asarray(dom, dtype=np.int64)].sum(axis=0), K)


def _compound_vs_itself(q_rot_group, k_rows, dom_fc, K):
    A = O.fc_scores_unit(q_rot_group, k_rows)
    s = A[np.asarray(list(dom_fc), dtype=np.int64)].sum(axis=0)
    return O.ca_from_scores(s, s, K)


def _dominant_set_skips_gaps(dom_row):
    return [int(i) for i in dom_row if int(i) >= 0]


def _dominant_set_sentinel_as_fc0(dom_row):
    return [max(int(i), 0) for i in dom_row]


def _fasa_m_values_by_length(n_layers, seq_len, d, n_tip, budget, bytes_per_param=2):
    d_dom = 2 * n_tip
    return float(n_layers * (seq_len * d_dom + budget * (d - d_dom) + seq_len * d) * bytes_per_param)


MUTATIONS = {
    "rope_row_vector_sign": ("rope_rotate", _rope_row_convention),
    "rope_rotate_half_pairing": ("rope_rotate", _rope_rotate_half),
    "tip_dropped_odd_term": ("fc_score", _fc_score_dropped_term),
    "fac_missing_sqrt_d": ("focused_attention_unit", _fac_unscaled),
    "topk_tie_to_larger_index": ("topk_select_unit", _topk_larger_index_first),
    "theta_exponent_halved": ("fc_frequencies", _freq_half_exponent),
    "kdom_splits_fc_pair": ("build_kdom", _kdom_wrong_pair),
    "gqa_modulo_mapping": ("focused_attention", _focused_attention_wrong_group),
    "append_rotates_one_position_late": ("append_token", _append_one_position_late),
    "ca_normalised_by_t": ("ca_from_scores", _ca_over_t),
    "calibration_keeps_lowest_ca": ("calibrate_dominant_fcs", _calibrate_lowest),
    "ca_compares_fc_with_itself": ("contextual_agreement_unit", _ca_fc_vs_itself),
    "compound_drops_last_fc": ("compound_agreement_unit", _compound_drops_last),
    "compound_compares_set_with_itself": ("compound_agreement_unit", _compound_vs_itself),
    "ragged_set_reads_past_the_sentinel": ("dominant_set", _dominant_set_skips_gaps),
    "ragged_sentinel_taken_as_fc0": ("dominant_set", _dominant_set_sentinel_as_fc0),
    "fasa_m_values_scale_with_length": ("fasa_m_gpu_bytes", _fasa_m_values_by_length),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    attr, fn = MUTATIONS[name]
    mod = _fresh_oracle()
    setattr(mod, attr, fn)
    failed = []
    for check in P.ALL_CHECKS:
        try:
            check(mod)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
