"""Comparison rules between the library and the oracle.

Tolerances (stated for this path):
  * TIP scores: |gpu - ref| <= 1e-3 * max(|ref|, RMS of ref over the row).
    (A strict relative test is meaningless for scores that cancel to ~0; the
    RMS floor keeps the bound relative to the row's scale.)
  * Selection: the index sets are equal except for tokens whose oracle score
    lies within 1e-3 (same floor) of the oracle's k-th largest score.
  * Attention output: relative L2 <= 2e-3 and max-abs <= 1e-2 for bf16 inputs;
    relative L2 <= 1e-5 and max-abs <= 1e-5 for fp32 inputs.
"""

import numpy as np

import oracle as O

TIP_RTOL = 1e-3
SEL_RTOL = 1e-3
OUT_TOL = {"bf16": (2e-3, 1e-2), "f32": (1e-5, 1e-5)}


def host_f64(t, dtype: str) -> np.ndarray:
    """Stored tensor (torch, any device) -> exact fp64 numpy."""
    import torch
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return O.decode_stored(t.view(torch.int16).numpy().view(np.uint16), "bf16")
    return O.decode_stored(t.numpy(), "f32")


def _floor(ref_row):
    ref_row = np.asarray(ref_row, dtype=np.float64)
    return np.sqrt(np.mean(ref_row ** 2)) if ref_row.size else 0.0


def check_scores(gpu_row, ref_row):
    gpu_row = np.asarray(gpu_row, dtype=np.float64)
    ref_row = np.asarray(ref_row, dtype=np.float64)
    bound = TIP_RTOL * np.maximum(np.abs(ref_row), _floor(ref_row))
    err = np.abs(gpu_row - ref_row)
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, f"{bad.size} TIP scores off, worst {np.max(err / np.maximum(bound, 1e-300)):.3g}x tol"


def check_selection(gpu_idx, ref_scores_row, k):
    """gpu_idx: the library's selected indices (count entries) for one unit."""
    s = np.asarray(ref_scores_row, dtype=np.float64)
    kk = min(k, s.shape[0])
    gpu = np.asarray(gpu_idx, dtype=np.int64)
    assert gpu.shape[0] == kk, f"count {gpu.shape[0]} != {kk}"
    assert np.all(np.diff(gpu) > 0), "indices not strictly ascending"
    assert gpu.min(initial=0) >= 0 and gpu.max(initial=0) < s.shape[0]
    ref = O.topk_select_unit(s, k)
    diff = np.setxor1d(gpu, ref)
    if diff.size:
        kth = np.sort(s)[::-1][kk - 1]
        tol = SEL_RTOL * max(abs(kth), _floor(s))
        far = diff[np.abs(s[diff] - kth) > tol]
        assert far.size == 0, f"{far.size} selected tokens differ beyond the near-tie band"
    return diff.size


def check_output(gpu, ref, dtype: str):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel_l2_tol, max_abs_tol = OUT_TOL[dtype]
    assert np.all(np.isfinite(gpu)), "non-finite output"
    rel = np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-300)
    mx = np.max(np.abs(gpu - ref)) if gpu.size else 0.0
    assert rel <= rel_l2_tol, f"rel-L2 {rel:.3g} > {rel_l2_tol}"
    assert mx <= max_abs_tol, f"max-abs {mx:.3g} > {max_abs_tol}"
    return rel, mx
