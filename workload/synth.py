"""Host-side (numpy) generator of the seeded synthetic FASA inputs.

Recipe (identical in ``csrc/synth_gen.cu``):

* Counter-based normals.  ``splitmix64`` is the SplitMix64 output function
  (Steele, Lea, Flood 2014).  A tensor stream has the base
  ``splitmix64((seed << 20) ^ (layer << 4) ^ tensor_id)`` with tensor ids
  Q=1, K=2, V=3; element ``i`` (row-major flat index) draws
  ``r1 = splitmix64(base + 2i)``, ``r2 = splitmix64(base + 2i + 1)``,
  ``u1 = ((r1 >> 11) + 1) / 2^53``, ``u2 = (r2 >> 11) / 2^53`` and the
  Box-Muller normal ``sqrt(-2 ln u1) cos(2 pi u2)``.
* Outlier FCs: per (layer, KV head) a seeded set of ``n_outlier`` frequency
  chunks; both dimensions of each are scaled x8 in the pre-RoPE key of that
  KV head and in the pre-RoPE query of every query head of its group.
* Dominant-FC table: per (layer, KV head) the outlier FCs plus a seeded
  uniform draw from the other FCs, ``n_tip`` in total, sorted ascending.
* Keys are stored post-RoPE: the key of token ``tau`` is rotated by
  ``tau * theta_i`` in each FC ``i`` (pairs ``(2i, 2i+1)``), with
  ``theta_i = rope_theta ** (-2i/d)``, computed in fp64 then rounded to the
  storage type.  Values and queries are stored as drawn (queries pre-RoPE).
* Lengths: the cache holds ``context`` tokens, or for a ragged workload
  ``len_b ~ U{lo..hi}`` seeded per sequence; the query sits at ``pos = len``.
* Storage: fp32, or bf16 by round-to-nearest-even from the fp32 value.
"""

import numpy as np

from .configs import Config

M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_G = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)

TENSOR_Q, TENSOR_K, TENSOR_V = 1, 2, 3
OUTLIER_SCALE = 8.0


def splitmix64(x):
    """SplitMix64 output function on uint64 (arrays or scalars), wrapping."""
    with np.errstate(over="ignore"):
        z = np.asarray(x, dtype=np.uint64) + _G
        z = (z ^ (z >> np.uint64(30))) * _C1
        z = (z ^ (z >> np.uint64(27))) * _C2
        return z ^ (z >> np.uint64(31))


def stream_base(seed: int, layer: int, tensor: int) -> np.uint64:
    key = (np.uint64(seed) << np.uint64(20)) ^ (np.uint64(layer) << np.uint64(4)) ^ np.uint64(tensor)
    return splitmix64(key)


def normals(base: np.uint64, start: int, count: int) -> np.ndarray:
    """Normals for flat indices start .. start+count-1 of one stream (fp64)."""
    i = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        r1 = splitmix64(base + np.uint64(2) * i)
        r2 = splitmix64(base + np.uint64(2) * i + np.uint64(1))
    u1 = ((r1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (r2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


def store(x64: np.ndarray, dtype: str) -> np.ndarray:
    x32 = x64.astype(np.float32)
    return x32 if dtype == "f32" else f32_to_bf16_bits(x32)


def outlier_fcs(cfg: Config, layer: int) -> np.ndarray:
    """[Hkv, n_outlier] int32, sorted per head."""
    out = np.zeros((cfg.n_kv_heads, cfg.n_outlier), dtype=np.int32)
    for h in range(cfg.n_kv_heads):
        rng = np.random.default_rng([cfg.seed, layer, h, 7])
        out[h] = np.sort(rng.choice(cfg.n_fc, cfg.n_outlier, replace=False))
    return out


def dominant_fcs(cfg: Config, layer: int, n_tip: int = None) -> np.ndarray:
    """[Hkv, n_tip] int32: the head's outlier FCs plus a seeded draw of others.
    With per-head counts, head h keeps its own count of FCs (drawn the same
    way) and the rest of its row is -1 (unused slots)."""
    if n_tip is None and cfg.n_tip_per_head is not None:
        out = np.full((cfg.n_kv_heads, cfg.n_tip), -1, dtype=np.int32)
        for h in range(cfg.n_kv_heads):
            n_h = cfg.n_tip_per_head[h]
            out[h, :n_h] = dominant_fcs(cfg, layer, n_h)[h]
        return out
    n_tip = cfg.n_tip if n_tip is None else n_tip
    outl = outlier_fcs(cfg, layer)
    dom = np.zeros((cfg.n_kv_heads, n_tip), dtype=np.int32)
    for h in range(cfg.n_kv_heads):
        keep = list(outl[h][: min(cfg.n_outlier, n_tip)])
        rest = np.setdiff1d(np.arange(cfg.n_fc), keep)
        rng = np.random.default_rng([cfg.seed, layer, h, 13])
        extra = rng.choice(rest, n_tip - len(keep), replace=False)
        dom[h] = np.sort(np.concatenate([np.asarray(keep, dtype=np.int64), extra]))
    return dom


def seq_lens(cfg: Config) -> np.ndarray:
    if cfg.ragged is None:
        return np.full(cfg.batch, cfg.context, dtype=np.int32)
    lo, hi = cfg.ragged
    rng = np.random.default_rng([cfg.seed, 11])
    return rng.integers(lo, hi + 1, size=cfg.batch).astype(np.int32)


def _fc_scale(cfg: Config, outl_h: np.ndarray) -> np.ndarray:
    s = np.ones(cfg.head_dim)
    for i in outl_h:
        s[2 * i] = s[2 * i + 1] = OUTLIER_SCALE
    return s


def gen_q(cfg: Config, layer: int = 0) -> np.ndarray:
    """Pre-RoPE queries [B, Hq, d] in fp64 (before storage rounding)."""
    d, G = cfg.head_dim, cfg.group
    outl = outlier_fcs(cfg, layer)
    q = normals(stream_base(cfg.seed, layer, TENSOR_Q), 0,
                cfg.batch * cfg.n_q_heads * d).reshape(cfg.batch, cfg.n_q_heads, d)
    for hq in range(cfg.n_q_heads):
        q[:, hq, :] *= _fc_scale(cfg, outl[hq // G])
    return q


def _key_rotation(cfg: Config, x: np.ndarray, positions: np.ndarray) -> np.ndarray:
    """Rotary encoding of stored keys: pair (2i, 2i+1) turned by tau*theta_i."""
    d = cfg.head_dim
    theta = cfg.rope_theta ** (-2.0 * np.arange(d // 2) / d)
    ang = positions[:, None].astype(np.float64) * theta[None, :]
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x0 * c - x1 * s
    y[..., 1::2] = x0 * s + x1 * c
    return y


def gen_kv_head(cfg: Config, layer: int, b: int, h: int, t_count: int = None):
    """Post-RoPE keys and values of one (b, KV head), fp64, [T, d] each."""
    d, T = cfg.head_dim, cfg.context
    t_count = T if t_count is None else t_count
    outl = outlier_fcs(cfg, layer)
    start = ((b * cfg.n_kv_heads + h) * T) * d
    kpre = normals(stream_base(cfg.seed, layer, TENSOR_K), start, t_count * d).reshape(t_count, d)
    kpre *= _fc_scale(cfg, outl[h])[None, :]
    k = _key_rotation(cfg, kpre, np.arange(t_count))
    v = normals(stream_base(cfg.seed, layer, TENSOR_V), start, t_count * d).reshape(t_count, d)
    return k, v


class LayerInputs:
    """Stored inputs of one attention layer (numpy, storage dtype)."""

    def __init__(self, cfg, q, k, v, dom_fc, lens):
        self.cfg = cfg
        self.q = q            # [B, Hq, d]  f32 or uint16 (bf16 bits), pre-RoPE
        self.k = k            # [B, Hkv, T, d] post-RoPE
        self.v = v            # [B, Hkv, T, d]
        self.dom_fc = dom_fc  # [Hkv, n] int32
        self.seq_lens = lens  # [B] int32
        self.pos = lens.copy()  # [B] int32, query right after the cache


def gen_layer(cfg: Config, layer: int = 0) -> LayerInputs:
    """All stored inputs of one layer on the host.  Sized for small/medium cases."""
    B, H, T, d = cfg.batch, cfg.n_kv_heads, cfg.context, cfg.head_dim
    st = np.float32 if cfg.dtype == "f32" else np.uint16
    k = np.empty((B, H, T, d), dtype=st)
    v = np.empty((B, H, T, d), dtype=st)
    for b in range(B):
        for h in range(H):
            kk, vv = gen_kv_head(cfg, layer, b, h)
            k[b, h] = store(kk, cfg.dtype)
            v[b, h] = store(vv, cfg.dtype)
    q = store(gen_q(cfg, layer), cfg.dtype)
    return LayerInputs(cfg, q, k, v, dominant_fcs(cfg, layer), seq_lens(cfg))
