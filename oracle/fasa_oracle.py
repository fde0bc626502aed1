"""fp64 CPU oracle of the FASA decode step (test infrastructure).

A plain, slow restatement of what the FASA pages define, written for a reader
to check against the text by eye.  All arithmetic is numpy fp64 on the host;
the inputs are the *stored* values (fp32, or bf16 bit patterns) promoted
exactly to fp64.  Only the tests, the smoke check and the benchmark's CPU
baseline use it; the CUDA library neither imports it nor is imported by it.

Sources (page title, then the section or equation):
  [P5] "FASA: Frequency-aware Sparse Attention", paper-graph-ui breakdown,
       §3.4 "RoPE from a Frequency-Chunk Perspective" (FC definition,
       theta_i = B^(-2i/d), the 2x2 rotation R_{m,theta_i}, the exact FC-wise
       decomposition of q R k^T), §3.4 "Online Stage 1: Token Importance
       Predictor (TIP)" (score S_t = sum over dominant FCs of alpha^(i);
       T_t = TopK-I(S_t, N_fac)), §3.4 "Online Stage 2: Focused Attention
       Computation (FAC)" (gather at original positions; softmax(q K_T^T /
       sqrt(d)) V_T), "Hardware-Aware Variants" (FASA-C, dominant key cache
       C_key^dom of t x 2 N_tip per head; Eq. 8 byte fraction).
  [P3] mlsanity.com "FASA: Frequency-aware Sparse Attention", abstract.

Readings where the pages are silent (each also listed in the design notes):
  * Keys in the cache are post-RoPE (FAC text: "the cached keys already
    encode their absolute positions"), so the query is rotated by its own
    position and TIP uses q' . k' per FC, which equals q R_{dt} k^T because
    R_m^T R_n = R_{n-m}.
  * FC i is the interleaved pair (2i, 2i+1); the rotation is applied to the
    column vector: (x0 cos a - x1 sin a, x0 sin a + x1 cos a).
  * GQA: one selection per (batch, KV head); the importance of a token is the
    sum over the G query heads of that group of their FC-restricted scores.
    Query head hq reads KV head hq // G.
  * TIP scores carry no 1/sqrt(d) (the page's S_t has none).
  * TopK-I ties: larger score first, equal scores -> smaller token index;
    the chosen indices are returned in ascending order; k' = min(k, len).
  * The cache holds tokens 0..len-1; the query is at position len unless the
    caller passes another position.

Parity pins for every function are in ``tests/test_oracle_pins.py``.
"""

import numpy as np

__all__ = [
    "decode_stored", "fc_frequencies", "rope_rotate", "apply_rope_q",
    "fc_score", "tip_scores_unit", "topk_select_unit", "focused_attention_unit",
    "tip_score", "topk_select", "focused_attention", "dense_attention",
    "decode_step", "append_token", "decode_step_append", "build_kdom", "bytes_fraction",
    "theoretical_speedup", "fc_scores_unit", "ca_from_scores", "contextual_agreement_unit",
    "calibrate_dominant_fcs", "compound_agreement_unit", "dominant_set", "fasa_m_gpu_bytes",
]


# ----------------------------------------------------------------------------
# Stored values -> fp64
# ----------------------------------------------------------------------------
def decode_stored(x, dtype: str) -> np.ndarray:
    """Promote stored fp32 values, or bf16 bit patterns (uint16), to fp64.

    bf16 is the upper half of an IEEE fp32 word, so shifting the 16 stored
    bits up by 16 gives the exact fp32 value.
    """
    x = np.asarray(x)
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        u = x.astype(np.uint16).astype(np.uint32) << np.uint32(16)
        return u.view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype}")


# ----------------------------------------------------------------------------
# RoPE, [P5] §3.4 "RoPE from a Frequency-Chunk Perspective"
# ----------------------------------------------------------------------------
def fc_frequencies(rope_theta: float, d: int) -> np.ndarray:
    """theta_i = B^(-2i/d) for FC i in 0 .. d/2-1."""
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(float(rope_theta), -2.0 * i / d)


def rope_rotate(x: np.ndarray, pos, rope_theta: float) -> np.ndarray:
    """Rotate every FC (x_2i, x_2i+1) of ``x`` [..., d] by pos * theta_i.

    ``pos`` broadcasts against x.shape[:-1].  R_{m,theta} =
    [[cos, -sin], [sin, cos]] applied to the column (x_2i, x_2i+1).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    theta = fc_frequencies(rope_theta, d)
    angle = np.asarray(pos, dtype=np.float64)[..., None] * theta
    c, s = np.cos(angle), np.sin(angle)
    out = np.empty_like(x)
    for i in range(d // 2):
        x0 = x[..., 2 * i]
        x1 = x[..., 2 * i + 1]
        out[..., 2 * i] = x0 * c[..., i] - x1 * s[..., i]
        out[..., 2 * i + 1] = x0 * s[..., i] + x1 * c[..., i]
    return out


def apply_rope_q(q: np.ndarray, pos: np.ndarray, rope_theta: float) -> np.ndarray:
    """q [B, Hq, d] (pre-RoPE, fp64), pos [B] -> rotated queries [B, Hq, d]."""
    q = np.asarray(q, dtype=np.float64)
    pos = np.asarray(pos, dtype=np.float64)
    return rope_rotate(q, pos[:, None], rope_theta)


# ----------------------------------------------------------------------------
# TIP, [P5] §3.4 "Online Stage 1: Token Importance Predictor (TIP)"
# ----------------------------------------------------------------------------
def fc_score(q_vec: np.ndarray, k_rows: np.ndarray, i: int) -> np.ndarray:
    """alpha^(i): the FC-i dot product of one rotated query with every key row."""
    return q_vec[2 * i] * k_rows[:, 2 * i] + q_vec[2 * i + 1] * k_rows[:, 2 * i + 1]


def tip_scores_unit(q_rot_group: np.ndarray, k_rows: np.ndarray, dom_fc) -> np.ndarray:
    """S over the cached tokens of one (batch, KV head).

    S_tau = sum_{g in group} sum_{i in I_dom} alpha_g^(i)(tau).
    ``q_rot_group`` [G, d], ``k_rows`` [len, d] (post-RoPE keys).
    """
    q_rot_group = np.atleast_2d(np.asarray(q_rot_group, dtype=np.float64))
    s = np.zeros(k_rows.shape[0], dtype=np.float64)
    for g in range(q_rot_group.shape[0]):
        for i in dom_fc:
            s += fc_score(q_rot_group[g], k_rows, int(i))
    return s


def topk_select_unit(scores: np.ndarray, k: int) -> np.ndarray:
    """T = TopK-I(S, k): indices of the min(k, len) largest scores.

    Stable ordering on (-score): equal scores keep token order, so the smaller
    index wins a tie (and -0 == +0).  Returned sorted ascending.
    """
    scores = np.asarray(scores, dtype=np.float64)
    kk = min(int(k), scores.shape[0])
    order = np.argsort(-scores, kind="stable")
    return np.sort(order[:kk]).astype(np.int64)


# ----------------------------------------------------------------------------
# FAC, [P5] §3.4 "Online Stage 2: Focused Attention Computation (FAC)"
# ----------------------------------------------------------------------------
def focused_attention_unit(q_rot_group, k_rows, v_rows, idx, return_weights=False):
    """O = softmax(q K_T^T / sqrt(d)) V_T over the gathered rows T = idx.

    Rows are gathered at their original positions (no re-indexing; the keys
    already carry their rotary encoding).  Returns [G, d] (and [G, |T|]).
    """
    q_rot_group = np.atleast_2d(np.asarray(q_rot_group, dtype=np.float64))
    d = q_rot_group.shape[1]
    idx = np.asarray(idx, dtype=np.int64)
    k_t = k_rows[idx]
    v_t = v_rows[idx]
    out = np.zeros((q_rot_group.shape[0], d), dtype=np.float64)
    weights = np.zeros((q_rot_group.shape[0], idx.shape[0]), dtype=np.float64)
    if idx.shape[0] == 0:
        return (out, weights) if return_weights else out
    for g in range(q_rot_group.shape[0]):
        logits = (k_t @ q_rot_group[g]) / np.sqrt(d)
        m = np.max(logits)
        w = np.exp(logits - m)
        w = w / np.sum(w)
        weights[g] = w
        out[g] = w @ v_t
    return (out, weights) if return_weights else out


# ----------------------------------------------------------------------------
# Whole-tensor stages (the library's C-ABI shapes)
# ----------------------------------------------------------------------------
def _group(n_q_heads: int, n_kv_heads: int) -> int:
    if n_q_heads % n_kv_heads:
        raise ValueError("n_q_heads must be a multiple of n_kv_heads")
    return n_q_heads // n_kv_heads


def dominant_set(dom_row) -> list:
    """I_dom of one KV head from its row of the dominant-FC table: the entries
    before the first negative one.  A negative entry marks an unused slot, so
    the heads of one layer may keep different numbers of FCs (the per-head
    N_tip the FASA pages propose under "Layer-wise and head-wise N_tip
    optimization"); a row without negative entries is used whole."""
    out = []
    for i in dom_row:
        if int(i) < 0:
            break
        out.append(int(i))
    return out


def tip_score(q_rot, K, dom_fc, seq_lens) -> np.ndarray:
    """q_rot [B,Hq,d], K [B,Hkv,T,d] fp64, dom_fc [Hkv,n] (per-head sets as
    dominant_set reads them), seq_lens [B] -> scores [B,Hkv,T] (NaN at
    tau >= len_b)."""
    B, Hq, d = q_rot.shape
    Hkv, T = K.shape[1], K.shape[2]
    G = _group(Hq, Hkv)
    out = np.full((B, Hkv, T), np.nan)
    for b in range(B):
        L = int(seq_lens[b])
        for h in range(Hkv):
            out[b, h, :L] = tip_scores_unit(q_rot[b, h * G:(h + 1) * G], K[b, h, :L], dominant_set(dom_fc[h]))
    return out


def topk_select(scores, seq_lens, k):
    """scores [B,Hkv,T] -> idx [B,Hkv,k] (ascending, -1 padded), count [B,Hkv]."""
    B, Hkv, _ = scores.shape
    idx = np.full((B, Hkv, k), -1, dtype=np.int64)
    count = np.zeros((B, Hkv), dtype=np.int64)
    for b in range(B):
        L = int(seq_lens[b])
        for h in range(Hkv):
            sel = topk_select_unit(scores[b, h, :L], k)
            idx[b, h, :sel.shape[0]] = sel
            count[b, h] = sel.shape[0]
    return idx, count


def focused_attention(q_rot, K, V, idx, count) -> np.ndarray:
    """FAC over the given index lists -> out [B,Hq,d]."""
    B, Hq, d = q_rot.shape
    Hkv = K.shape[1]
    G = _group(Hq, Hkv)
    out = np.zeros((B, Hq, d))
    for b in range(B):
        for h in range(Hkv):
            sel = np.asarray(idx[b, h, :int(count[b, h])], dtype=np.int64)
            out[b, h * G:(h + 1) * G] = focused_attention_unit(
                q_rot[b, h * G:(h + 1) * G], K[b, h], V[b, h], sel)
    return out


def dense_attention(q_rot, K, V, seq_lens) -> np.ndarray:
    """Full-KV decode attention: FAC with T = all cached tokens 0..len-1."""
    B, Hkv = K.shape[0], K.shape[1]
    idx = [[np.arange(int(seq_lens[b])) for _ in range(Hkv)] for b in range(B)]
    cnt = np.array([[int(seq_lens[b])] * Hkv for b in range(B)])
    T = K.shape[2]
    full = np.full((B, Hkv, T), -1, dtype=np.int64)
    for b in range(B):
        for h in range(Hkv):
            full[b, h, :cnt[b, h]] = idx[b][h]
    return focused_attention(q_rot, K, V, full, cnt)


def decode_step(q, pos, K, V, dom_fc, seq_lens, k, rope_theta):
    """One FASA decode step: RoPE(q) -> TIP -> TopK-I -> FAC.

    q [B,Hq,d] pre-RoPE fp64, pos [B], K/V [B,Hkv,T,d] fp64 (keys post-RoPE),
    dom_fc [Hkv,n], seq_lens [B], budget k.  Returns (out [B,Hq,d],
    idx [B,Hkv,k], count [B,Hkv], scores [B,Hkv,T]).
    """
    q_rot = apply_rope_q(q, pos, rope_theta)
    scores = tip_score(q_rot, K, dom_fc, seq_lens)
    idx, count = topk_select(scores, seq_lens, k)
    out = focused_attention(q_rot, K, V, idx, count)
    return out, idx, count, scores


def append_token(K, V, k_new, v_new, seq_lens, rope_theta):
    """The new token of a decode step enters the cache: its key, rotated by
    its own position len_b (keys are cached post-RoPE), and its value go to
    index len_b.  K/V [B,Hkv,T,d] fp64 (copied), k_new/v_new [B,Hkv,d] fp64
    (k_new pre-RoPE).  Returns (K', V', seq_lens + 1)."""
    K = np.array(K, dtype=np.float64, copy=True)
    V = np.array(V, dtype=np.float64, copy=True)
    lens = np.asarray(seq_lens, dtype=np.int64)
    for b in range(K.shape[0]):
        t = int(lens[b])
        K[b, :, t, :] = rope_rotate(np.asarray(k_new[b], dtype=np.float64), t, rope_theta)
        V[b, :, t, :] = np.asarray(v_new[b], dtype=np.float64)
    return K, V, lens + 1


def decode_step_append(q, k_new, v_new, K, V, dom_fc, seq_lens, k, rope_theta):
    """A decode step that first appends the new token (``append_token``) and
    then attends over len_b + 1 tokens with the query at position len_b, the
    new token's own position.  Returns decode_step's tuple plus (K', V')."""
    K2, V2, lens2 = append_token(K, V, k_new, v_new, seq_lens, rope_theta)
    res = decode_step(q, np.asarray(seq_lens), K2, V2, dom_fc, lens2, k, rope_theta)
    return res + (K2, V2)


def build_kdom(K_stored: np.ndarray, dom_fc: np.ndarray, block: int = 64) -> np.ndarray:
    """Dominant key cache C_key^dom of stored values, FC-major within blocks of
    `block` tokens: [B, Hkv, T/block, n, block, 2].

    K_dom[b,h,t//block,j,t%block,:] = K[b,h,t, 2*dom_fc[h,j] : 2*dom_fc[h,j]+2]
    (a copy; the FC pair is never split).  Unused slots (negative entries)
    hold zeros here; the library leaves them untouched.
    """
    B, Hkv, T, _ = K_stored.shape
    n = dom_fc.shape[1]
    out = np.zeros((B, Hkv, T // block, n, block, 2), dtype=K_stored.dtype)
    for h in range(Hkv):
        for j in range(n):
            i = int(dom_fc[h, j])
            if i < 0:
                continue
            cols = K_stored[:, h, :, 2 * i:2 * i + 2]           # [B, T, 2]
            out[:, h, :, j, :, :] = cols.reshape(B, T // block, block, 2)
    return out


# ----------------------------------------------------------------------------
# Contextual Agreement and the offline calibration, [P5] "The Functional
# Sparsity Hypothesis and the Contextual Agreement (CA) Metric" (Eq. 4) and
# the calibration objective with its procedure (Algorithm 1)
# ----------------------------------------------------------------------------
def fc_scores_unit(q_rot_group: np.ndarray, k_rows: np.ndarray) -> np.ndarray:
    """Single-FC scores of every FC i for one (batch, KV head):
    alpha_i[tau] = sum over the group's query heads of q'^[i] . k_tau^[i]
    (post-RoPE, the same group sum as TIP).  Returns [d/2, t]."""
    q = np.asarray(q_rot_group, dtype=np.float64)
    K = np.asarray(k_rows, dtype=np.float64)
    F = K.shape[1] // 2
    return np.stack([fc_score(q[g], K, i) for i in range(F) for g in range(q.shape[0])]
                    ).reshape(F, q.shape[0], -1).sum(axis=1)


def ca_from_scores(full: np.ndarray, alpha_i: np.ndarray, K: int) -> float:
    """Eq. 4: |TopK-I(full, K) & TopK-I(alpha_i, K)| / K, with K' = min(K, t)
    in place of K (both sets hold every token when t <= K)."""
    t = len(full)
    kk = min(K, t)
    if kk == 0:
        return 1.0
    a = set(topk_select_unit(full, kk).tolist())
    b = set(topk_select_unit(alpha_i, kk).tolist())
    return len(a & b) / kk


def contextual_agreement_unit(q_rot_group, k_rows, K: int) -> np.ndarray:
    """CA of every FC for one (batch, KV head) and one query group: the full
    head's scores are the sum of the single-FC scores (the FC decomposition
    of q R k^T).  Returns [d/2]; all ones when no token is cached."""
    if np.asarray(k_rows).shape[0] == 0:
        return np.ones(np.asarray(k_rows).shape[1] // 2)
    A = fc_scores_unit(q_rot_group, k_rows)
    full = A.sum(axis=0)
    return np.array([ca_from_scores(full, A[i], K) for i in range(A.shape[0])])


def compound_agreement_unit(q_rot_group, k_rows, dom_fc, K: int) -> float:
    """Compound CA of a chosen FC set I_dom for one (batch, KV head): Eq. 4
    with alpha_i replaced by the summed scores of the chosen FCs -- the
    statistic the CA page reports for the dominant sets (its Table 1), and
    the TIP score S of the same set -- against the full head's scores.
    1 when no token is cached."""
    if np.asarray(k_rows).shape[0] == 0:
        return 1.0
    A = fc_scores_unit(q_rot_group, k_rows)
    full = A.sum(axis=0)
    chosen = A[np.asarray(dominant_set(dom_fc), dtype=np.int64)].sum(axis=0)
    return ca_from_scores(full, chosen, K)


def calibrate_dominant_fcs(ca_mean: np.ndarray, n_tip: int) -> np.ndarray:
    """Algorithm 1, last step: per head, the n_tip FCs with the highest mean
    CA (equal means: smaller FC index first), returned in ascending order.
    ca_mean [Hkv, d/2] -> [Hkv, n_tip] int32."""
    ca_mean = np.asarray(ca_mean, dtype=np.float64)
    out = np.empty((ca_mean.shape[0], n_tip), dtype=np.int32)
    for h in range(ca_mean.shape[0]):
        order = np.argsort(-ca_mean[h], kind="stable")[:n_tip]
        out[h] = np.sort(order)
    return out


# ----------------------------------------------------------------------------
# Byte model, [P5] "Hardware-Aware Variants", FASA-C and Eq. 8
# ----------------------------------------------------------------------------
def bytes_fraction(n_tip: int, d: int, budget: int, t: int) -> float:
    """Fraction of a full K+V read that FASA-C loads per step.

    TIP reads t x d_dom elements (d_dom = 2 N_tip), FAC reads 2 N_fac d, full
    attention reads 2 t d:  (t d_dom + 2 N_fac d) / (2 t d).
    """
    d_dom = 2 * n_tip
    return (t * d_dom + 2 * budget * d) / (2.0 * t * d)


def fasa_m_gpu_bytes(n_layers: int, seq_len: int, d: int, n_tip: int, budget: int,
                     bytes_per_param: int = 2) -> float:
    """Eq. 10 ("Hardware-Aware Variants", FASA-M): GPU memory per head of the
    memory-optimised variant,
        N_layers x (L d_dom + b d_nondom + b d) x bytes_per_param,
    d_dom = 2 N_tip, d_nondom = d - d_dom, b = N_fac: the dominant keys of
    every token, plus the selected tokens' other key dimensions and values."""
    d_dom = 2 * n_tip
    return float(n_layers * (seq_len * d_dom + budget * (d - d_dom) + budget * d) * bytes_per_param)


def theoretical_speedup(n_tip: int, d: int, budget: int, t: int) -> float:
    """Eq. 8: 2 t d / (2 t N_tip + 2 N_fac d)."""
    return (2.0 * t * d) / (2.0 * t * n_tip + 2.0 * budget * d)
