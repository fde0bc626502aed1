"""ctypes binding of libfasa.so.

Each function has the name of its C entry point and takes torch CUDA tensors
(or raw device addresses as ints).  It checks dtypes and contiguity, passes
``data_ptr()`` and the current CUDA stream, and raises ``FasaError`` on a
non-zero status.  Nothing here computes on the data.
"""

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(PKG, "libfasa.so")

FASA_F32, FASA_BF16 = 0, 1
FASA_DEV_BAD_INPUT, FASA_DEV_TIMEOUT, FASA_DEV_UNDRAINED = 1, 2, 4

EXPORTS = [
    "fasa_version", "fasa_status_string", "fasa_last_cuda_error", "fasa_max_budget",
    "fasa_workspace_size", "fasa_apply_rope_q", "fasa_build_kdom", "fasa_append_kdom",
    "fasa_tip_score", "fasa_topk_select", "fasa_focused_attention", "fasa_dense_attention",
    "fasa_decode_step", "fasa_device_status", "fasa_cluster_size", "fasa_decode_step_noalloc",
    "fasa_decode_step_append", "fasa_fc_agreement_workspace_size", "fasa_fc_agreement",
    "fasa_select_dominant_fcs", "fasa_compound_agreement", "fasa_test_fault_injection", "fasa_step_kernel",
    "fasa_build_knondom", "fasa_decode_step_split", "fasa_decode_step_append_split",
]


class FasaError(RuntimeError):
    def __init__(self, fn, status, lib):
        msg = lib.fasa_status_string(status).decode()
        if status == 4:
            msg += f" (cudaError {lib.fasa_last_cuda_error()})"
        super().__init__(f"{fn}: {msg}")
        self.status = status


class FasaDims(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("t_max", ctypes.c_int32), ("n_tip", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32), ("rope_theta", ctypes.c_double),
    ]


def dims_for(cfg, cluster_ctas: int = 0, **override) -> FasaDims:
    """FasaDims from a workload config (anything with the same field names)."""
    d = dict(batch=cfg.batch, n_q_heads=cfg.n_q_heads, n_kv_heads=cfg.n_kv_heads,
             head_dim=cfg.head_dim, t_max=cfg.context, n_tip=cfg.n_tip,
             dtype=FASA_F32 if cfg.dtype == "f32" else FASA_BF16, rope_theta=cfg.rope_theta)
    d.update(override)
    return FasaDims(d["batch"], d["n_q_heads"], d["n_kv_heads"], d["head_dim"], d["t_max"],
                    d["n_tip"], d["dtype"], cluster_ctas, float(d["rope_theta"]))


_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib():
    """Load libfasa.so once.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "`python -m kv_cache_token_tip_gb300.build` (there is no fallback)")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        dp = ctypes.POINTER(FasaDims)
        sig = {
            "fasa_version": ([], ctypes.c_int),
            "fasa_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "fasa_last_cuda_error": ([], ctypes.c_int),
            "fasa_max_budget": ([dp, ctypes.POINTER(i32)], ctypes.c_int),
            "fasa_workspace_size": ([dp, i32, ctypes.POINTER(sz)], ctypes.c_int),
            "fasa_cluster_size": ([dp, ctypes.POINTER(i32)], ctypes.c_int),
            "fasa_step_kernel": ([dp, ctypes.POINTER(i32)], ctypes.c_int),
            "fasa_apply_rope_q": ([vp, vp, vp, dp, vp], ctypes.c_int),
            "fasa_build_kdom": ([vp, vp, vp, vp, dp, vp], ctypes.c_int),
            "fasa_build_knondom": ([vp, vp, vp, vp, dp, vp], ctypes.c_int),
            "fasa_decode_step_split": ([vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, dp, vp],
                                       ctypes.c_int),
            "fasa_append_kdom": ([vp, vp, vp, vp, dp, vp], ctypes.c_int),
            "fasa_tip_score": ([vp, vp, vp, vp, vp, dp, vp], ctypes.c_int),
            "fasa_topk_select": ([vp, vp, i32, vp, vp, dp, vp], ctypes.c_int),
            "fasa_focused_attention": ([vp, vp, vp, vp, vp, vp, i32, vp, dp, vp], ctypes.c_int),
            "fasa_dense_attention": ([vp, vp, vp, vp, vp, dp, vp], ctypes.c_int),
            "fasa_decode_step": ([vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, dp, vp],
                                 ctypes.c_int),
            "fasa_device_status": ([vp, ctypes.POINTER(i32)], ctypes.c_int),
            "fasa_decode_step_noalloc": ([vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, dp, vp], ctypes.c_int),
            "fasa_decode_step_append": ([vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, dp, vp],
                                        ctypes.c_int),
            "fasa_decode_step_append_split": ([vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, sz, dp, vp],
                                              ctypes.c_int),
            "fasa_fc_agreement_workspace_size": ([dp, ctypes.POINTER(sz)], ctypes.c_int),
            "fasa_fc_agreement": ([vp, vp, vp, i32, vp, vp, sz, dp, vp], ctypes.c_int),
            "fasa_compound_agreement": ([vp, vp, vp, vp, i32, vp, vp, sz, dp, vp], ctypes.c_int),
            "fasa_select_dominant_fcs": ([vp, i32, vp, dp, vp], ctypes.c_int),
            "fasa_test_fault_injection": ([ctypes.c_uint64, i32, i32], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


# ---------------------------------------------------------------- marshalling
def _ptr(x, dtype=None, name="tensor", host_ok=False):
    """Device pointer of a contiguous tensor.  With host_ok, a tensor in pinned
    host memory is accepted too (the GPU reads or writes it in place over the
    host link: the FASA-M placement of the K/V caches, zero-copy step I/O)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    import torch
    if not x.is_cuda and not (host_ok and x.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor" + (" or pinned host memory" if host_ok else ""))
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and x.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {x.dtype}, expected {dtype}")
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _store_dtypes():
    import torch
    return (torch.float32, torch.bfloat16)


def _check(fn, st):
    if st != 0:
        raise FasaError(fn, st, lib())


def _i32():
    import torch
    return torch.int32


def _f32():
    import torch
    return torch.float32


# ---------------------------------------------------------------- entry points
def fasa_max_budget(dims: FasaDims) -> int:
    out = ctypes.c_int32(0)
    _check("fasa_max_budget", lib().fasa_max_budget(ctypes.byref(dims), ctypes.byref(out)))
    return out.value


def fasa_workspace_size(dims: FasaDims, budget: int) -> int:
    out = ctypes.c_size_t(0)
    _check("fasa_workspace_size", lib().fasa_workspace_size(ctypes.byref(dims), budget, ctypes.byref(out)))
    return out.value


def fasa_cluster_size(dims: FasaDims) -> int:
    out = ctypes.c_int32(0)
    _check("fasa_cluster_size", lib().fasa_cluster_size(ctypes.byref(dims), ctypes.byref(out)))
    return out.value


FASA_KERNEL_CLUSTER, FASA_KERNEL_SINGLE_EXCHANGE = 0, 1


def fasa_step_kernel(dims: FasaDims) -> int:
    """Which fused kernel serves fasa_decode_step for these dims on this
    device (FASA_KERNEL_CLUSTER or FASA_KERNEL_SINGLE_EXCHANGE)."""
    out = ctypes.c_int32(0)
    _check("fasa_step_kernel", lib().fasa_step_kernel(ctypes.byref(dims), ctypes.byref(out)))
    return out.value


def fasa_apply_rope_q(q, pos, q_rot, dims: FasaDims, stream=None):
    _check("fasa_apply_rope_q", lib().fasa_apply_rope_q(
        _ptr(q, _store_dtypes(), "q"), _ptr(pos, _i32(), "pos"), _ptr(q_rot, _f32(), "q_rot"),
        ctypes.byref(dims), _stream(stream)))


def fasa_build_kdom(k_cache, dom_fc, seq_lens, k_dom, dims: FasaDims, stream=None):
    _check("fasa_build_kdom", lib().fasa_build_kdom(
        _ptr(k_cache, _store_dtypes(), "k_cache"), _ptr(dom_fc, _i32(), "dom_fc"),
        _ptr(seq_lens, _i32(), "seq_lens"), _ptr(k_dom, _store_dtypes(), "k_dom"),
        ctypes.byref(dims), _stream(stream)))


def fasa_build_knondom(k_cache, dom_fc, seq_lens, k_nondom, dims: FasaDims, stream=None):
    """The non-dominant key pairs of every token, in FC order (FASA-M split
    keys); k_cache and k_nondom may live in page-locked host memory."""
    _check("fasa_build_knondom", lib().fasa_build_knondom(
        _ptr(k_cache, _store_dtypes(), "k_cache", True), _ptr(dom_fc, _i32(), "dom_fc"),
        _ptr(seq_lens, _i32(), "seq_lens"), _ptr(k_nondom, _store_dtypes(), "k_nondom", True),
        ctypes.byref(dims), _stream(stream)))


def fasa_decode_step_split(q, pos, k_nondom, v_cache, k_dom, dom_fc, seq_lens, budget: int, out,
                           idx_out=None, count_out=None, workspace=None, dims: FasaDims = None, stream=None):
    """fasa_decode_step with the keys split: non-dominant pairs in k_nondom,
    dominant ones in k_dom (FASA-M)."""
    ws_bytes = 0
    if workspace is not None and not isinstance(workspace, int):
        ws_bytes = workspace.numel() * workspace.element_size()
    _check("fasa_decode_step_split", lib().fasa_decode_step_split(
        _ptr(q, _store_dtypes(), "q", True), _ptr(pos, _i32(), "pos", True),
        _ptr(k_nondom, _store_dtypes(), "k_nondom", True), _ptr(v_cache, _store_dtypes(), "v_cache", True),
        _ptr(k_dom, _store_dtypes(), "k_dom"), _ptr(dom_fc, _i32(), "dom_fc"),
        _ptr(seq_lens, _i32(), "seq_lens", True), int(budget), _ptr(out, _f32(), "out", True),
        _ptr(idx_out, _i32(), "idx_out", True), _ptr(count_out, _i32(), "count_out", True),
        _ptr(workspace, None, "workspace"), ws_bytes, ctypes.byref(dims), _stream(stream)))


def fasa_append_kdom(k_new, dom_fc, tok_pos, k_dom, dims: FasaDims, stream=None):
    _check("fasa_append_kdom", lib().fasa_append_kdom(
        _ptr(k_new, _store_dtypes(), "k_new"), _ptr(dom_fc, _i32(), "dom_fc"),
        _ptr(tok_pos, _i32(), "tok_pos"), _ptr(k_dom, _store_dtypes(), "k_dom"),
        ctypes.byref(dims), _stream(stream)))


def fasa_tip_score(q_rot, k_dom, dom_fc, seq_lens, scores, dims: FasaDims, stream=None):
    _check("fasa_tip_score", lib().fasa_tip_score(
        _ptr(q_rot, _f32(), "q_rot"), _ptr(k_dom, _store_dtypes(), "k_dom"),
        _ptr(dom_fc, _i32(), "dom_fc"), _ptr(seq_lens, _i32(), "seq_lens"),
        _ptr(scores, _f32(), "scores"), ctypes.byref(dims), _stream(stream)))


def fasa_topk_select(scores, seq_lens, budget: int, idx, count, dims: FasaDims, stream=None):
    _check("fasa_topk_select", lib().fasa_topk_select(
        _ptr(scores, _f32(), "scores"), _ptr(seq_lens, _i32(), "seq_lens"), int(budget),
        _ptr(idx, _i32(), "idx"), _ptr(count, _i32(), "count"), ctypes.byref(dims), _stream(stream)))


def fasa_focused_attention(q_rot, k_cache, v_cache, seq_lens, idx, count, budget: int, out,
                           dims: FasaDims, stream=None):
    _check("fasa_focused_attention", lib().fasa_focused_attention(
        _ptr(q_rot, _f32(), "q_rot"), _ptr(k_cache, _store_dtypes(), "k_cache", True),
        _ptr(v_cache, _store_dtypes(), "v_cache", True), _ptr(seq_lens, _i32(), "seq_lens"),
        _ptr(idx, _i32(), "idx"), _ptr(count, _i32(), "count"), int(budget),
        _ptr(out, _f32(), "out"), ctypes.byref(dims), _stream(stream)))


def fasa_dense_attention(q_rot, k_cache, v_cache, seq_lens, out, dims: FasaDims, stream=None):
    _check("fasa_dense_attention", lib().fasa_dense_attention(
        _ptr(q_rot, _f32(), "q_rot"), _ptr(k_cache, _store_dtypes(), "k_cache", True),
        _ptr(v_cache, _store_dtypes(), "v_cache", True), _ptr(seq_lens, _i32(), "seq_lens"),
        _ptr(out, _f32(), "out"), ctypes.byref(dims), _stream(stream)))


def fasa_decode_step(q, pos, k_cache, v_cache, k_dom, dom_fc, seq_lens, budget: int, out,
                     idx_out=None, count_out=None, workspace=None, dims: FasaDims = None, stream=None):
    ws_bytes = 0
    if workspace is not None and not isinstance(workspace, int):
        ws_bytes = workspace.numel() * workspace.element_size()
    _check("fasa_decode_step", lib().fasa_decode_step(
        _ptr(q, _store_dtypes(), "q", True), _ptr(pos, _i32(), "pos", True),
        _ptr(k_cache, _store_dtypes(), "k_cache", True), _ptr(v_cache, _store_dtypes(), "v_cache", True),
        _ptr(k_dom, _store_dtypes(), "k_dom"), _ptr(dom_fc, _i32(), "dom_fc"),
        _ptr(seq_lens, _i32(), "seq_lens", True), int(budget), _ptr(out, _f32(), "out", True),
        _ptr(idx_out, _i32(), "idx_out", True), _ptr(count_out, _i32(), "count_out", True),
        _ptr(workspace, None, "workspace"), ws_bytes, ctypes.byref(dims), _stream(stream)))


def fasa_decode_step_append(q, k_new, v_new, seq_lens, k_cache, v_cache, k_dom, dom_fc, budget: int, out,
                            idx_out=None, count_out=None, workspace=None, dims: FasaDims = None, stream=None):
    """The decode step with the new token appended first: k_new (pre-RoPE)
    and v_new [B,Hkv,d] go to index seq_lens[b] of the caches (and K_dom),
    and the step attends over seq_lens[b] + 1 tokens with the query at
    position seq_lens[b].  seq_lens is not advanced."""
    ws_bytes = 0
    if workspace is not None and not isinstance(workspace, int):
        ws_bytes = workspace.numel() * workspace.element_size()
    _check("fasa_decode_step_append", lib().fasa_decode_step_append(
        _ptr(q, _store_dtypes(), "q"), _ptr(k_new, _store_dtypes(), "k_new"),
        _ptr(v_new, _store_dtypes(), "v_new"), _ptr(seq_lens, _i32(), "seq_lens"),
        _ptr(k_cache, _store_dtypes(), "k_cache", True), _ptr(v_cache, _store_dtypes(), "v_cache", True),
        _ptr(k_dom, _store_dtypes(), "k_dom"), _ptr(dom_fc, _i32(), "dom_fc"), int(budget),
        _ptr(out, _f32(), "out"), _ptr(idx_out, _i32(), "idx_out"), _ptr(count_out, _i32(), "count_out"),
        _ptr(workspace, None, "workspace"), ws_bytes, ctypes.byref(dims), _stream(stream)))


def fasa_decode_step_append_split(q, k_new, v_new, seq_lens, k_nondom, v_cache, k_dom, dom_fc, budget: int, out,
                                  idx_out=None, count_out=None, workspace=None, dims: FasaDims = None, stream=None):
    """fasa_decode_step_append over split keys: the new token's non-dominant
    pairs go to its k_nondom row, its dominant pairs to K_dom, v_new to
    v_cache; then the split step attends over seq_lens[b] + 1 tokens."""
    ws_bytes = 0
    if workspace is not None and not isinstance(workspace, int):
        ws_bytes = workspace.numel() * workspace.element_size()
    _check("fasa_decode_step_append_split", lib().fasa_decode_step_append_split(
        _ptr(q, _store_dtypes(), "q"), _ptr(k_new, _store_dtypes(), "k_new"),
        _ptr(v_new, _store_dtypes(), "v_new"), _ptr(seq_lens, _i32(), "seq_lens"),
        _ptr(k_nondom, _store_dtypes(), "k_nondom", True), _ptr(v_cache, _store_dtypes(), "v_cache", True),
        _ptr(k_dom, _store_dtypes(), "k_dom"), _ptr(dom_fc, _i32(), "dom_fc"), int(budget),
        _ptr(out, _f32(), "out"), _ptr(idx_out, _i32(), "idx_out"), _ptr(count_out, _i32(), "count_out"),
        _ptr(workspace, None, "workspace"), ws_bytes, ctypes.byref(dims), _stream(stream)))


def fasa_fc_agreement_workspace_size(dims: FasaDims) -> int:
    out = ctypes.c_size_t(0)
    _check("fasa_fc_agreement_workspace_size",
           lib().fasa_fc_agreement_workspace_size(ctypes.byref(dims), ctypes.byref(out)))
    return out.value


def fasa_fc_agreement(q_rot, k_cache, seq_lens, topk: int, ca, dims: FasaDims, workspace=None, stream=None):
    """Contextual Agreement of every FC for every (batch, KV head):
    ca [B, Hkv, d/2] fp32.  Without a workspace one is allocated here."""
    if workspace is None:
        import torch
        workspace = torch.empty(fasa_fc_agreement_workspace_size(dims), dtype=torch.uint8, device=ca.device)
    _check("fasa_fc_agreement", lib().fasa_fc_agreement(
        _ptr(q_rot, _f32(), "q_rot"), _ptr(k_cache, _store_dtypes(), "k_cache"),
        _ptr(seq_lens, _i32(), "seq_lens"), int(topk), _ptr(ca, _f32(), "ca"),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(), ctypes.byref(dims),
        _stream(stream)))


def fasa_compound_agreement(q_rot, k_cache, dom_fc, seq_lens, topk: int, cca, dims: FasaDims, workspace=None,
                            stream=None):
    """Compound CA of the chosen FCs dom_fc [Hkv, n_tip] per (batch, KV head):
    cca [B, Hkv] fp32.  Without a workspace one is allocated here."""
    if workspace is None:
        import torch
        workspace = torch.empty(fasa_fc_agreement_workspace_size(dims), dtype=torch.uint8, device=cca.device)
    _check("fasa_compound_agreement", lib().fasa_compound_agreement(
        _ptr(q_rot, _f32(), "q_rot"), _ptr(k_cache, _store_dtypes(), "k_cache"), _ptr(dom_fc, _i32(), "dom_fc"),
        _ptr(seq_lens, _i32(), "seq_lens"), int(topk), _ptr(cca, _f32(), "cca"),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(), ctypes.byref(dims),
        _stream(stream)))


def fasa_select_dominant_fcs(ca_mean, n_tip: int, dom_fc, dims: FasaDims, stream=None):
    """dom_fc [Hkv, n_tip] int32 <- the n_tip FCs of highest mean CA per head."""
    _check("fasa_select_dominant_fcs", lib().fasa_select_dominant_fcs(
        _ptr(ca_mean, _f32(), "ca_mean"), int(n_tip), _ptr(dom_fc, _i32(), "dom_fc"), ctypes.byref(dims),
        _stream(stream)))


def fasa_decode_step_noalloc(q, pos, k_cache, v_cache, k_dom, dom_fc, seq_lens, budget: int, out,
                             idx_out=None, count_out=None, dims: FasaDims = None, stream=None):
    """fasa_decode_step without a workspace argument: for callers that cannot
    allocate device memory, the step uses the library's fixed scratch array."""
    _check("fasa_decode_step_noalloc", lib().fasa_decode_step_noalloc(
        _ptr(q, _store_dtypes(), "q"), _ptr(pos, _i32(), "pos"),
        _ptr(k_cache, _store_dtypes(), "k_cache", True), _ptr(v_cache, _store_dtypes(), "v_cache", True),
        _ptr(k_dom, _store_dtypes(), "k_dom"), _ptr(dom_fc, _i32(), "dom_fc"),
        _ptr(seq_lens, _i32(), "seq_lens"), int(budget), _ptr(out, _f32(), "out"),
        _ptr(idx_out, _i32(), "idx_out"), _ptr(count_out, _i32(), "count_out"),
        ctypes.byref(dims), _stream(stream)))


def fasa_device_status(stream=None) -> int:
    out = ctypes.c_int32(0)
    _check("fasa_device_status", lib().fasa_device_status(_stream(stream), ctypes.byref(out)))
    return out.value


def fasa_test_fault_injection(wait_limit_ns: int = 1_000_000_000, drop_tip_tile: int = -1,
                              drop_fac_refill: int = -1) -> None:
    """Test hook: bound of every device wait, one TIP tile whose copy the
    fused step never issues, and one refill of the single-exchange kernel's
    FAC whose completion is never reported (-1: none).  The defaults restore
    normal runs."""
    _check("fasa_test_fault_injection", lib().fasa_test_fault_injection(int(wait_limit_ns), int(drop_tip_tile),
                                                                         int(drop_fac_refill)))
