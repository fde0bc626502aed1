"""Device-side synthetic inputs: the same recipe as ``synth.py``, drawn on the
GPU by ``libfasa_synth.so`` (built from ``csrc/synth_gen.cu``).

Returns torch CUDA tensors; the host tables (outlier FCs, dominant FCs,
lengths) come from ``synth.py``.
"""

import ctypes
import os

import numpy as np

from . import synth
from .configs import Config

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfasa_synth.so")
_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} missing: run `python -m kv_cache_token_tip_gb300.build`")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i = ctypes.c_void_p, ctypes.c_int
        L.synth_fill_layer.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_double,
                                       ctypes.c_ulonglong, i, i, vp]
        L.synth_fill_layer.restype = ctypes.c_int
        _lib = L
    return _lib


def torch_dtype(cfg: Config):
    import torch
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


class DeviceLayer:
    """One layer's stored inputs on the GPU plus the host tables."""

    def __init__(self, cfg, q, k, v, dom_fc, seq_lens, pos):
        self.cfg = cfg
        self.q, self.k, self.v = q, k, v          # storage dtype
        self.dom_fc, self.seq_lens, self.pos = dom_fc, seq_lens, pos   # int32 CUDA
        self.dom_fc_host = dom_fc.cpu().numpy()
        self.seq_lens_host = seq_lens.cpu().numpy()
        self.pos_host = pos.cpu().numpy()


def alloc_layer(cfg: Config, device="cuda"):
    import torch
    dt = torch_dtype(cfg)
    B, Hq, H, T, d = cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.context, cfg.head_dim
    q = torch.empty((B, Hq, d), dtype=dt, device=device)
    k = torch.empty((B, H, T, d), dtype=dt, device=device)
    v = torch.empty((B, H, T, d), dtype=dt, device=device)
    return q, k, v


def fill_layer(cfg: Config, layer: int, q, k, v, stream=None):
    """Draw layer `layer` of `cfg` into the given tensors (on `stream`)."""
    import torch
    outl = torch.from_numpy(synth.outlier_fcs(cfg, layer).astype(np.int32)).to(q.device)
    s = torch.cuda.current_stream() if stream is None else stream
    rc = _load().synth_fill_layer(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), outl.data_ptr(), cfg.n_outlier, cfg.batch,
        cfg.n_q_heads, cfg.n_kv_heads, cfg.context, cfg.head_dim, float(cfg.rope_theta),
        cfg.seed, layer, 0 if cfg.dtype == "f32" else 1, s.cuda_stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_layer failed: cudaError {rc}")
    s.synchronize()   # keeps `outl` alive until the kernel is done


def make_layer(cfg: Config, layer: int = 0, device="cuda") -> DeviceLayer:
    import torch
    q, k, v = alloc_layer(cfg, device)
    fill_layer(cfg, layer, q, k, v)
    dom = torch.from_numpy(synth.dominant_fcs(cfg, layer).astype(np.int32)).to(device)
    lens = torch.from_numpy(synth.seq_lens(cfg).astype(np.int32)).to(device)
    return DeviceLayer(cfg, q, k, v, dom, lens, lens.clone())


def upload_layer(inp: "synth.LayerInputs", device="cuda") -> DeviceLayer:
    """Host-generated inputs (synth.gen_layer) copied to the device."""
    import torch
    cfg = inp.cfg

    def up(x):
        if cfg.dtype == "f32":
            return torch.from_numpy(np.ascontiguousarray(x)).to(device)
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(device).view(torch.bfloat16)

    dom = torch.from_numpy(inp.dom_fc.astype(np.int32)).to(device)
    lens = torch.from_numpy(inp.seq_lens.astype(np.int32)).to(device)
    pos = torch.from_numpy(inp.pos.astype(np.int32)).to(device)
    return DeviceLayer(cfg, up(inp.q), up(inp.k), up(inp.v), dom, lens, pos)
