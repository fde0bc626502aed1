"""Pins of the fp64 oracle: facts the FASA pages and the mathematics fix.

Each ``check_*`` takes the oracle module (so a test can hand it a copy with a
planted mistake) and raises AssertionError when the pin does not hold.  None
of them retypes the oracle's own formula: each compares against an
independent statement of the same fact (a closed form, a library routine, a
brute-force enumeration, an invariant or a number the pages print).
"""

import itertools
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# --- P2: RoPE -----------------------------------------------------------------
def check_rope_complex_closed_form(o):
    """R_{m,theta_i} acting on (x_2i, x_2i+1) is multiplication of the complex
    number x_2i + i x_2i+1 by exp(i m theta_i), with theta_i = B^(-2i/d)
    written as exp(-(2i/d) ln B)."""
    rng = _rng(1)
    for d, base in ((8, 1e4), (64, 1e4), (128, 5e5)):
        x = rng.standard_normal((5, d))
        pos = np.array([0, 1, 17, 1024, 131072])
        y = o.rope_rotate(x, pos, base)
        theta = np.exp(-(2.0 * np.arange(d // 2) / d) * np.log(base))
        z = (x[:, 0::2] + 1j * x[:, 1::2]) * np.exp(1j * pos[:, None] * theta[None, :])
        assert np.allclose(y[:, 0::2], z.real, rtol=0, atol=1e-9), "RoPE even dims"
        assert np.allclose(y[:, 1::2], z.imag, rtol=0, atol=1e-9), "RoPE odd dims"


def check_rope_norm_and_relative(o):
    """Each FC keeps its norm; (R_m q).(R_n k) depends only on m - n."""
    rng = _rng(2)
    d, base = 128, 1e6
    q = rng.standard_normal(d)
    k = rng.standard_normal(d)
    for m in (0, 5, 4096):
        qm = o.rope_rotate(q, m, base)
        assert np.allclose(qm[0::2] ** 2 + qm[1::2] ** 2, q[0::2] ** 2 + q[1::2] ** 2,
                           rtol=1e-12, atol=1e-12), "RoPE changed an FC norm"
    for (m, n, s) in ((10, 3, 100), (4096, 4000, 7), (1, 0, 30000)):
        a = np.dot(o.rope_rotate(q, m, base), o.rope_rotate(k, n, base))
        b = np.dot(o.rope_rotate(q, m + s, base), o.rope_rotate(k, n + s, base))
        assert abs(a - b) <= 1e-9 * (1 + abs(a)), "score depends on absolute position"
    # q R_{dt} k^T with the block-diagonal R of the pages: rotating q by m and
    # k by n gives the pre-RoPE pair rotated by the relative angle.
    m, n = 777, 123
    lhs = np.dot(o.rope_rotate(q, m, base), o.rope_rotate(k, n, base))
    theta = np.exp(-(2.0 * np.arange(d // 2) / d) * np.log(base))
    qc = q[0::2] + 1j * q[1::2]
    kc = k[0::2] + 1j * k[1::2]
    rhs = np.sum((qc * np.conj(kc) * np.exp(1j * (m - n) * theta)).real)
    assert abs(lhs - rhs) <= 1e-9 * (1 + abs(rhs)), "relative-position form"


def check_fc_frequencies(o):
    """theta_0 = 1, theta_i strictly decreasing (low FC index = high
    frequency), constant ratio B^(2/d), theta_{d/2} would be 1/B."""
    for d, base in ((64, 1e4), (128, 5e5)):
        th = o.fc_frequencies(base, d)
        assert th.shape == (d // 2,)
        assert th[0] == 1.0
        assert np.all(np.diff(th) < 0)
        r = th[:-1] / th[1:]
        assert np.allclose(r, base ** (2.0 / d), rtol=1e-12)
        assert np.isclose(th[-1] / base ** (2.0 / d), 1.0 / base, rtol=1e-12)


def check_rope_matches_cached_key_convention(o):
    """The oracle's query rotation and the generator's stored-key rotation use
    one convention: q'_m . k'_n equals the relative-angle complex form."""
    from workload import configs, synth
    cfg = configs.CONFIGS["tiny_fp32_ctx1k"].with_(context=64)
    kk, _ = synth.gen_kv_head(cfg, 0, 0, 0, t_count=64)   # post-RoPE keys, fp64
    rng = _rng(3)
    d = cfg.head_dim
    q = rng.standard_normal(d)
    m = 64
    qr = o.rope_rotate(q, m, cfg.rope_theta)
    # undo the key rotation independently through the complex form
    theta = np.exp(-(2.0 * np.arange(d // 2) / d) * np.log(cfg.rope_theta))
    for n in (0, 1, 33, 63):
        kc_post = kk[n, 0::2] + 1j * kk[n, 1::2]
        kc_pre = kc_post * np.exp(-1j * n * theta)
        qc = q[0::2] + 1j * q[1::2]
        rhs = np.sum((qc * np.conj(kc_pre) * np.exp(1j * (m - n) * theta)).real)
        assert abs(np.dot(qr, kk[n]) - rhs) <= 1e-9 * (1 + abs(rhs))


# --- P1 / P3: the FC decomposition is exact -----------------------------------
def check_all_fcs_equal_full_logits(o):
    """With I_dom = all d/2 FCs, S = q.K^T exactly (G = 1), and for a GQA group
    S = (sum_g q_g).K^T (the score is linear in the query)."""
    rng = _rng(4)
    d = 64
    K = rng.standard_normal((50, d))
    q = rng.standard_normal((1, d))
    s = o.tip_scores_unit(q, K, np.arange(d // 2))
    assert np.allclose(s, K @ q[0], rtol=1e-12, atol=1e-12), "sum over all FCs != full dot"
    qg = rng.standard_normal((3, d))
    s = o.tip_scores_unit(qg, K, np.arange(d // 2))
    assert np.allclose(s, K @ qg.sum(0), rtol=1e-12, atol=1e-11)


def check_fc_additivity(o):
    """Scores over a partition of the FCs add up to the score over their union."""
    rng = _rng(5)
    d = 128
    K = rng.standard_normal((40, d))
    q = rng.standard_normal((4, d))
    perm = rng.permutation(d // 2)
    parts = [perm[:5], perm[5:20], perm[20:21], perm[21:]]
    total = sum(o.tip_scores_unit(q, K, p) for p in parts)
    assert np.allclose(total, K @ q.sum(0), rtol=1e-12, atol=1e-11)
    # restricting to FCs touches exactly the pair (2i, 2i+1): zeroing every
    # other dimension of K does not change the restricted score
    dom = perm[:7]
    mask = np.zeros(d)
    mask[2 * dom] = 1
    mask[2 * dom + 1] = 1
    assert np.allclose(o.tip_scores_unit(q, K, dom), (K * mask) @ q.sum(0), rtol=1e-12, atol=1e-11)


def check_dom_order_invariance(o):
    """S is a sum over a set: the order of I_dom does not matter (P9)."""
    rng = _rng(6)
    K = rng.standard_normal((30, 64))
    q = rng.standard_normal((2, 64))
    dom = np.array([3, 17, 4, 30, 9])
    a = o.tip_scores_unit(q, K, dom)
    b = o.tip_scores_unit(q, K, dom[::-1])
    assert np.allclose(a, b, rtol=1e-13, atol=1e-13)


# --- P5 / P6 / P9: TopK-I ------------------------------------------------------
def check_topk_bruteforce(o):
    """TopK-I equals the max-sum subset of size k, ties resolved to the
    lexicographically smallest index set (= smaller index first)."""
    rng = _rng(7)
    for trial in range(60):
        n = int(rng.integers(1, 10))
        k = int(rng.integers(1, 12))
        s = rng.integers(-3, 4, size=n).astype(np.float64)   # many ties
        if trial % 3 == 0:
            s = rng.standard_normal(n)
        kk = min(k, n)
        best = None
        for sub in itertools.combinations(range(n), kk):
            val = s[list(sub)].sum()
            key = (-val, sub)
            if best is None or key < best:
                best = key
        got = o.topk_select_unit(s, k)
        assert tuple(int(x) for x in got) == best[1], (s, k, got, best)


def check_topk_batched_layout(o):
    """The batched TopK-I: each (batch, KV head) row holds the brute-force
    best set of min(k, len) tokens (ties to the smaller index) in ascending
    order, then -1; count = min(k, len); an empty sequence selects nothing."""
    rng = _rng(83)
    B, H, T, k = 3, 2, 9, 4
    scores = rng.integers(-2, 3, size=(B, H, T)).astype(np.float64)
    lens = np.array([9, 3, 0])
    idx, cnt = o.topk_select(scores, lens, k)
    assert idx.shape == (B, H, k) and cnt.shape == (B, H)
    for b in range(B):
        for h in range(H):
            L = int(lens[b])
            kk = min(k, L)
            assert cnt[b, h] == kk
            best = min(itertools.combinations(range(L), kk), key=lambda sub: (-scores[b, h, list(sub)].sum(), sub))
            assert tuple(int(x) for x in idx[b, h, :kk]) == best
            assert np.all(idx[b, h, kk:] == -1)


def check_fac_subset_vs_sdpa(o):
    """FAC over index subsets equals torch's scaled_dot_product_attention over
    the gathered rows, with query head hq reading KV head hq // G."""
    import torch
    rng = _rng(89)
    B, Hq, Hkv, T, d, k = 2, 6, 3, 25, 32, 7
    q = rng.standard_normal((B, Hq, d))
    K = rng.standard_normal((B, Hkv, T, d))
    V = rng.standard_normal((B, Hkv, T, d))
    idx = np.full((B, Hkv, k), -1, dtype=np.int64)
    cnt = np.zeros((B, Hkv), dtype=np.int64)
    for b in range(B):
        for h in range(Hkv):
            c = int(rng.integers(1, k + 1))
            idx[b, h, :c] = np.sort(rng.choice(T, c, replace=False))
            cnt[b, h] = c
    out = o.focused_attention(q, K, V, idx, cnt)
    G = Hq // Hkv
    for b in range(B):
        for hq in range(Hq):
            h = hq // G
            sel = idx[b, h, :cnt[b, h]]
            qt = torch.from_numpy(q[b, hq][None, None, :])
            kt = torch.from_numpy(K[b, h, sel][None])
            vt = torch.from_numpy(V[b, h, sel][None])
            ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0, 0].numpy()
            assert np.allclose(out[b, hq], ref, rtol=1e-12, atol=1e-12)


def check_topk_signed_zero_and_order(o):
    """-0 and +0 are equal scores; output is ascending; k >= len keeps all."""
    s = np.array([0.0, -0.0, 1.0, -0.0, 0.0])
    assert list(o.topk_select_unit(s, 3)) == [0, 1, 2]
    s = np.array([5.0, 1.0, 7.0, 3.0])
    assert list(o.topk_select_unit(s, 2)) == [0, 2]
    assert list(o.topk_select_unit(s, 10)) == [0, 1, 2, 3]


def check_topk_permutation(o):
    """Permuting tie-free scores permutes the selected set the same way."""
    rng = _rng(8)
    s = rng.standard_normal(200)
    perm = rng.permutation(200)
    a = set(int(x) for x in o.topk_select_unit(s, 17))
    b = set(int(perm[x]) for x in o.topk_select_unit(s[perm], 17))
    assert a == b


def check_query_scale_invariance(o):
    """Scaling the query by c > 0 scales every S by c: the selection is unchanged."""
    rng = _rng(9)
    K = rng.standard_normal((300, 64))
    q = rng.standard_normal((2, 64))
    dom = np.array([1, 5, 9, 20])
    a = o.topk_select_unit(o.tip_scores_unit(q, K, dom), 20)
    b = o.topk_select_unit(o.tip_scores_unit(3.7 * q, K, dom), 20)
    assert np.array_equal(a, b)


# --- P4 / P6 / P7: FAC ---------------------------------------------------------
def check_fac_weights(o):
    """Weights are >= 0 and sum to 1 over T; rows outside T get no weight
    (changing them leaves the output unchanged); the output is a convex
    combination of the selected value rows."""
    rng = _rng(10)
    d = 64
    K = rng.standard_normal((80, d))
    V = rng.standard_normal((80, d))
    q = rng.standard_normal((3, d)) * 3
    idx = np.array([2, 9, 10, 40, 79])
    out, w = o.focused_attention_unit(q, K, V, idx, return_weights=True)
    assert np.all(w >= 0) and np.allclose(w.sum(1), 1.0, atol=1e-12)
    K2, V2 = K.copy(), V.copy()
    others = np.setdiff1d(np.arange(80), idx)
    K2[others] = 1e3
    V2[others] = -1e3
    assert np.allclose(o.focused_attention_unit(q, K2, V2, idx), out, atol=1e-12)
    lo, hi = V[idx].min(0), V[idx].max(0)
    assert np.all(out >= lo - 1e-12) and np.all(out <= hi + 1e-12)


def check_fac_single_token(o):
    """k = 1: the output is exactly the value row of the top-scored token."""
    rng = _rng(11)
    K = rng.standard_normal((64, 32))
    V = rng.standard_normal((64, 32))
    q = rng.standard_normal((2, 32))
    s = o.tip_scores_unit(q, K, np.arange(16))
    sel = o.topk_select_unit(s, 1)
    assert sel[0] == int(np.argmax(s))
    out = o.focused_attention_unit(q, K, V, sel)
    assert np.array_equal(out, np.stack([V[sel[0]]] * 2))


def check_fac_vs_sdpa(o):
    """Dense attention (T = all tokens) equals torch's scaled_dot_product_attention
    in fp64 on the CPU, including the GQA mapping hq -> hq // G."""
    import torch
    rng = _rng(12)
    B, Hq, Hkv, T, d = 2, 6, 2, 37, 64
    q = rng.standard_normal((B, Hq, d))
    K = rng.standard_normal((B, Hkv, T, d))
    V = rng.standard_normal((B, Hkv, T, d))
    lens = np.array([37, 20])
    out = o.dense_attention(q, K, V, lens)
    G = Hq // Hkv
    for b in range(B):
        L = lens[b]
        qt = torch.from_numpy(q[b][:, None, :])                               # [Hq,1,d]
        kt = torch.from_numpy(np.repeat(K[b, :, :L], G, axis=0))              # [Hq,L,d]
        vt = torch.from_numpy(np.repeat(V[b, :, :L], G, axis=0))
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[:, 0].numpy()
        assert np.allclose(out[b], ref, rtol=1e-12, atol=1e-12)


def check_full_budget_equals_dense(o):
    """All FCs dominant and budget = len: the FASA step equals dense attention
    of the rotated query (the pages' correctness guarantee with nothing
    evicted), and the TIP scores equal the summed full logits."""
    import torch
    rng = _rng(13)
    B, Hq, Hkv, T, d, base = 1, 4, 2, 48, 64, 1e4
    q = rng.standard_normal((B, Hq, d))
    K = rng.standard_normal((B, Hkv, T, d))
    V = rng.standard_normal((B, Hkv, T, d))
    lens = np.array([T])
    pos = np.array([T])
    dom = np.tile(np.arange(d // 2), (Hkv, 1))
    out, idx, cnt, sc = o.decode_step(q, pos, K, V, dom, lens, T, base)
    assert int(cnt[0, 0]) == T and np.array_equal(idx[0, 0], np.arange(T))
    # independent rotation through the complex form, then SDPA
    theta = np.exp(-(2.0 * np.arange(d // 2) / d) * np.log(base))
    z = (q[..., 0::2] + 1j * q[..., 1::2]) * np.exp(1j * T * theta)
    qr = np.empty_like(q)
    qr[..., 0::2], qr[..., 1::2] = z.real, z.imag
    G = Hq // Hkv
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qr[0][:, None, :]),
        torch.from_numpy(np.repeat(K[0], G, axis=0)),
        torch.from_numpy(np.repeat(V[0], G, axis=0)))[:, 0].numpy()
    assert np.allclose(out[0], ref, rtol=1e-11, atol=1e-11)
    for h in range(Hkv):
        assert np.allclose(sc[0, h], K[0, h] @ qr[0, h * G:(h + 1) * G].sum(0), rtol=1e-11, atol=1e-10)


def check_gqa_mapping(o):
    """Query head hq attends to KV head hq // G: with every value row of KV
    head h equal to h + 1, the output of head hq is hq // G + 1."""
    rng = _rng(14)
    B, Hq, Hkv, T, d = 2, 8, 2, 40, 64
    q = rng.standard_normal((B, Hq, d))
    K = rng.standard_normal((B, Hkv, T, d))
    V = np.zeros((B, Hkv, T, d))
    for h in range(Hkv):
        V[:, h] = h + 1
    dom = np.tile(np.arange(4), (Hkv, 1))
    out, _, _, _ = o.decode_step(q, np.array([T, T]), K, V, dom, np.array([T, 25]), 7, 1e4)
    for hq in range(Hq):
        assert np.allclose(out[:, hq], hq // (Hq // Hkv) + 1, atol=1e-12)


def check_decode_stored(o):
    """bf16 bit patterns promote exactly (torch's bfloat16 -> float64 agrees)."""
    import torch
    rng = _rng(15)
    x = torch.from_numpy(rng.standard_normal(1000).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(o.decode_stored(bits, "bf16"), x.to(torch.float64).numpy())
    f = rng.standard_normal(10).astype(np.float32)
    assert np.array_equal(o.decode_stored(f, "f32"), f.astype(np.float64))


def check_build_kdom_layout(o):
    """K_dom is FC-major within token blocks: K_dom[b,h,t//4,j,t%4,c] holds
    K[b,h,t,2 dom[h,j] + c].  Keys that encode their own coordinates make the
    layout self-evident."""
    B, H, T, d = 2, 3, 12, 16
    K = np.zeros((B, H, T, d), dtype=np.float32)
    for b in range(B):
        for h in range(H):
            for t in range(T):
                K[b, h, t] = b * 1e6 + h * 1e4 + t * 100 + np.arange(d)
    dom = np.array([[0, 5, 7], [1, 2, 3], [7, 6, 0]])
    kd = o.build_kdom(K, dom, block=4)
    assert kd.shape == (B, H, 3, 3, 4, 2)
    assert kd[1, 2, 1, 0, 0, 1] == 1e6 + 2e4 + 400 + 15   # t=4, FC 7 -> dims 14, 15
    assert kd[0, 0, 2, 1, 1, 0] == 900 + 10               # t=9, FC 5 -> dim 10
    assert kd[1, 1, 0, 2, 0, 0] == 1e6 + 1e4 + 6          # t=0, FC 3 -> dim 6
    assert kd[0, 1, 2, 0, 3, 1] == 1e4 + 1100 + 3         # t=11, FC 1 -> dim 3


def check_byte_model(o):
    """The numbers the pages print for the FASA-C memory-movement model."""
    with open(os.path.join(GOLDEN, "byte_model.json")) as f:
        g = json.load(f)["cases"]
    c = g[0]
    assert abs(o.bytes_fraction(c["n_tip"], c["d"], c["budget"], c["t"]) - c["fraction"]) <= c["abs_tol"]
    c = g[1]
    assert np.isclose(o.bytes_fraction(c["n_tip"], c["d"], 0, 10 ** 6), c["tip_fraction"], rtol=1e-12)
    c = g[2]
    assert np.isclose(o.theoretical_speedup(c["n_tip"], c["d"], 0, 10 ** 6), c["speedup_limit"], rtol=1e-12)
    assert o.theoretical_speedup(c["n_tip"], c["d"], 256, 10 ** 9) < c["speedup_limit"]
    c = g[3]
    assert abs(c["t"] / c["budget"] - c["fac_ratio_approx"]) / c["fac_ratio_approx"] <= c["rel_tol"]


# --- NEXT-1: appending the step's own token ---------------------------------
def check_append_same_position_dot(o):
    """The new key is rotated by its own position, which is also the query's
    position: R_m^T R_m = I makes every FC's rotated dot q'.k' equal the
    pre-RoPE dot q.k."""
    rng = _rng(41)
    B, Hkv, T, d = 2, 2, 12, 8
    K = rng.standard_normal((B, Hkv, T, d))
    V = rng.standard_normal((B, Hkv, T, d))
    k_new = rng.standard_normal((B, Hkv, d))
    v_new = rng.standard_normal((B, Hkv, d))
    q = rng.standard_normal((B, Hkv, d))          # one query head per KV head
    lens = np.array([5, 11])
    K2, V2, lens2 = o.append_token(K, V, k_new, v_new, lens, 1e4)
    assert np.array_equal(lens2, lens + 1)
    qr = o.apply_rope_q(q, lens, 1e4)
    for b in range(B):
        t = lens[b]
        for h in range(Hkv):
            for i in range(d // 2):
                lhs = qr[b, h, 2 * i] * K2[b, h, t, 2 * i] + qr[b, h, 2 * i + 1] * K2[b, h, t, 2 * i + 1]
                rhs = q[b, h, 2 * i] * k_new[b, h, 2 * i] + q[b, h, 2 * i + 1] * k_new[b, h, 2 * i + 1]
                assert abs(lhs - rhs) <= 1e-12 * (1 + abs(rhs))
        assert np.array_equal(V2[b, :, t], v_new[b])
        keep = np.ones(T, dtype=bool)
        keep[t] = False
        assert np.array_equal(K2[b][:, keep], K[b][:, keep]) and np.array_equal(V2[b][:, keep], V[b][:, keep])


def check_append_empty_cache(o):
    """With an empty cache the step attends over its own token only: every
    query head's output is its KV head's new value."""
    rng = _rng(42)
    B, Hkv, G, T, d = 2, 2, 3, 4, 8
    K = np.zeros((B, Hkv, T, d))
    V = np.zeros((B, Hkv, T, d))
    q = rng.standard_normal((B, Hkv * G, d))
    k_new = rng.standard_normal((B, Hkv, d))
    v_new = rng.standard_normal((B, Hkv, d))
    dom = np.array([[0, 2], [1, 3]])
    out, idx, cnt, _, _, _ = o.decode_step_append(q, k_new, v_new, K, V, dom, np.array([0, 0]), 4, 1e4)
    assert np.all(cnt == 1) and np.all(idx[:, :, 0] == 0)
    for b in range(B):
        for hq in range(Hkv * G):
            assert np.allclose(out[b, hq], v_new[b, hq // G], atol=1e-14)


def check_append_equals_cached_token(o):
    """Appending equals a plain step over a cache that already holds the
    token, its key rotated here by the complex-exponential closed form
    (x0 + i x1) e^{i t theta_j}."""
    rng = _rng(43)
    B, Hkv, G, T, d, theta = 1, 2, 2, 20, 8, 1e4
    K = rng.standard_normal((B, Hkv, T, d))
    V = rng.standard_normal((B, Hkv, T, d))
    q = rng.standard_normal((B, Hkv * G, d))
    k_new = rng.standard_normal((B, Hkv, d))
    v_new = rng.standard_normal((B, Hkv, d))
    dom = np.array([[0, 3], [1, 2]])
    lens = np.array([13])
    out, idx, cnt, sc, _, _ = o.decode_step_append(q, k_new, v_new, K, V, dom, lens, 6, theta)
    Kc, Vc = K.copy(), V.copy()
    t = int(lens[0])
    for h in range(Hkv):
        z = (k_new[0, h, 0::2] + 1j * k_new[0, h, 1::2]) * np.exp(1j * t * theta ** (-np.arange(d // 2) * 2.0 / d))
        Kc[0, h, t, 0::2], Kc[0, h, t, 1::2] = z.real, z.imag
        Vc[0, h, t] = v_new[0, h]
    out2, idx2, cnt2, _ = o.decode_step(q, lens, Kc, Vc, dom, lens + 1, 6, theta)
    assert np.array_equal(idx, idx2) and np.array_equal(cnt, cnt2)
    assert np.allclose(out, out2, rtol=1e-12, atol=1e-12)


# --- NEXT-4: Contextual Agreement (Eq. 4) and calibration (Algorithm 1) -----
def check_ca_hand_examples(o):
    """Overlaps worked out by hand (TopK-I: larger first, ties to the smaller
    token index)."""
    full = np.array([6.0, 5, 4, 3, 2, 1])                  # top-3: {0, 1, 2}
    assert o.ca_from_scores(full, np.array([1.0, 2, 3, 6, 5, 4]), 3) == 0.0       # {3, 4, 5}
    assert abs(o.ca_from_scores(full, np.array([6.0, 1, 5, 2, 4, 3]), 3) - 2 / 3) < 1e-15  # {0, 2, 4}
    assert o.ca_from_scores(full, full * 7.0, 3) == 1.0     # same ranking
    ties_full = np.array([1.0, 1, 1, 0])                    # top-2: {0, 1}
    assert o.ca_from_scores(ties_full, np.array([0.0, 1, 1, 1]), 2) == 0.5  # {1, 2}
    assert o.ca_from_scores(full, -full, 6) == 1.0          # K = t: every token in both


def check_ca_bounds_and_short_contexts(o):
    rng = _rng(51)
    q = rng.standard_normal((3, 8))
    K = rng.standard_normal((40, 8))
    ca = o.contextual_agreement_unit(q, K, 7)
    assert ca.shape == (4,) and np.all((ca >= 0) & (ca <= 1))
    assert np.all(np.abs(ca * 7 - np.round(ca * 7)) < 1e-12)  # multiples of 1/K
    assert np.all(o.contextual_agreement_unit(q, K[:5], 7) == 1.0)  # t <= K


def check_ca_single_carrying_fc(o):
    """A query whose only non-zero FC is j: FC j's scores are the full scores
    (CA 1); every other FC scores all tokens 0, so its top-K is the first K
    tokens and its CA is the share of the full top-K below index K."""
    rng = _rng(52)
    t, K, j = 50, 6, 2
    q = np.zeros((2, 8))
    q[:, 2 * j:2 * j + 2] = rng.standard_normal((2, 2))
    Kr = rng.standard_normal((t, 8))
    ca = o.contextual_agreement_unit(q, Kr, K)
    full = Kr @ q.sum(axis=0)
    top = sorted(range(t), key=lambda tau: (-full[tau], tau))[:K]
    share = sum(1 for tau in top if tau < K) / K
    assert ca[j] == 1.0
    for i in range(4):
        if i != j:
            assert ca[i] == share


def check_fc_scores_sum_to_logits(o):
    rng = _rng(53)
    q = rng.standard_normal((4, 16))
    K = rng.standard_normal((30, 16))
    A = o.fc_scores_unit(q, K)
    assert A.shape == (8, 30)
    assert np.allclose(A.sum(axis=0), K @ q.sum(axis=0), rtol=1e-12, atol=1e-12)
    assert np.allclose(A[3], K[:, 6:8] @ q[:, 6:8].sum(axis=0), rtol=1e-12, atol=1e-12)


def check_calibration_selection(o):
    ca = np.array([[0.1, 0.5, 0.5, 0.2], [0.9, 0.1, 0.3, 0.3], [0.3, 0.3, 0.3, 0.3]])
    assert np.array_equal(o.calibrate_dominant_fcs(ca, 2), [[1, 2], [0, 2], [0, 1]])
    assert np.array_equal(o.calibrate_dominant_fcs(ca, 3), [[1, 2, 3], [0, 2, 3], [0, 1, 2]])


def check_ca_without_tokens(o):
    """Nothing cached: both TopK-I sets are empty, read as full agreement."""
    q = _rng(59).standard_normal((2, 8))
    K = np.zeros((0, 8))
    assert np.array_equal(o.contextual_agreement_unit(q, K, 4), np.ones(4))
    assert o.compound_agreement_unit(q, K, [1, 2], 4) == 1.0


def check_compound_all_fcs_is_one(o):
    """Choosing every FC sums to the full logits: the two sets coincide."""
    rng = _rng(61)
    q = rng.standard_normal((3, 16))
    K = rng.standard_normal((40, 16))
    for k in (1, 5, 40, 100):
        assert o.compound_agreement_unit(q, K, range(8), k) == 1.0


def check_compound_single_fc_is_ca(o):
    """A one-FC set is Eq. 4 itself; a set missing the FC that carries the
    logits agrees less than the set holding it."""
    rng = _rng(67)
    q = rng.standard_normal((3, 16))
    K = rng.standard_normal((40, 16))
    ca = o.contextual_agreement_unit(q, K, 5)
    for i in range(8):
        assert o.compound_agreement_unit(q, K, [i], 5) == ca[i]
    assert len(set(ca.tolist())) > 1   # the pin distinguishes the FCs
    # FC 3 carries the logits (x20): every set holding it reaches 1 here
    K2 = K.copy()
    K2[:, 6:8] *= 20.0
    q2 = q.copy()
    q2[:, 6:8] *= 20.0
    assert o.compound_agreement_unit(q2, K2, [1, 3, 5], 5) == 1.0
    assert o.compound_agreement_unit(q2, K2, [0, 1, 2, 4, 5, 6, 7], 5) < 1.0


def check_compound_scores_are_tip_scores(o):
    """The chosen set's summed scores are the TIP scores of that set."""
    rng = _rng(71)
    q = rng.standard_normal((4, 16))
    K = rng.standard_normal((50, 16))
    dom = [0, 3, 6]
    full = K @ q.sum(axis=0)
    S = o.tip_scores_unit(q, K, dom)
    for k in (3, 10):
        expect = len(set(o.topk_select_unit(full, k).tolist()) & set(o.topk_select_unit(S, k).tolist())) / k
        assert o.compound_agreement_unit(q, K, dom, k) == expect


# --- per-head ragged N_tip ---------------------------------------------------
def check_dominant_set_reading(o):
    assert o.dominant_set([3, 5, -1, -1]) == [3, 5]
    assert o.dominant_set([1, -1, 2]) == [1]
    assert o.dominant_set([-1, 2]) == []
    assert o.dominant_set(np.array([4, 0, 7], dtype=np.int32)) == [4, 0, 7]


def check_ragged_tip_closed_form(o):
    """Heads keeping 1 and 3 FCs: each head's scores are its own FCs' query
    columns (group-summed) times the key columns -- a matrix product."""
    rng = _rng(73)
    B, Hq, Hkv, T, d = 1, 4, 2, 20, 16
    q = rng.standard_normal((B, Hq, d))
    K = rng.standard_normal((B, Hkv, T, d))
    dom = np.array([[5, -1, -1], [0, 2, 7]], dtype=np.int32)
    s = o.tip_score(q, K, dom, np.array([T]))
    for h, fcs in ((0, [5]), (1, [0, 2, 7])):
        cols = np.concatenate([[2 * i, 2 * i + 1] for i in fcs])
        qbar = q[0, 2 * h:2 * h + 2].sum(axis=0)
        assert np.allclose(s[0, h], K[0, h][:, cols] @ qbar[cols], rtol=1e-12, atol=1e-12)


def check_ragged_kdom_slots(o):
    K = _rng(79).standard_normal((1, 2, 64, 8))
    kd = o.build_kdom(K, np.array([[3, -1], [1, 2]], dtype=np.int32))
    assert np.array_equal(kd[0, 0, 0, 0], K[0, 0, :, 6:8])
    assert np.all(kd[0, 0, 0, 1] == 0)
    assert np.array_equal(kd[0, 1, 0, 1], K[0, 1, :, 4:6])


def check_fasa_m_memory(o):
    """Eq. 10 against the page's worked example (tests/golden/fasa_m_memory.json):
    d_dom = 0.25 d and b = 0.1 L give 0.25 + 0.075 + 0.1 = 0.425 L d per head,
    about 4.7x below the 2 L d of a full cache."""
    with open(os.path.join(GOLDEN, "fasa_m_memory.json")) as f:
        c0, c1 = json.load(f)["cases"]
    L, d, n, b = c0["seq_len"], c0["d"], c0["n_tip"], c0["budget"]
    assert 2 * n == c0["dominant_coef"] * d and b == c0["values_coef"] * L
    per_head = o.fasa_m_gpu_bytes(1, L, d, n, b, bytes_per_param=1)
    assert abs(per_head - c0["total_coef"] * L * d) < 1e-9 * L * d
    parts = (c0["dominant_coef"], c0["nondominant_coef"], c0["values_coef"])
    assert abs(sum(parts) - c0["total_coef"]) < 1e-12
    assert abs(c1["full_coef"] / c0["total_coef"] - c1["reduction_approx"]) <= c1["abs_tol"]
    # layers and element size scale it linearly; no budget leaves the dominant keys
    assert o.fasa_m_gpu_bytes(32, L, d, n, b, 2) == 64 * per_head
    assert o.fasa_m_gpu_bytes(1, L, d, n, 0, 1) == L * 2 * n


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
