"""The bounded device waits of the fused step (GPU).

A step whose TIP stage barrier is armed for a copy that is never issued
(fasa_test_fault_injection) must end by itself once the wait bound runs out,
report FASA_DEV_TIMEOUT in the device status word, and leave the stream and
the context usable: the next step, with the defaults restored, gives the
same result as a step before the fault.  Nothing here faults the GPU: the
wait that runs out is on a shared-memory barrier no copy targets.
"""

import time

import numpy as np
import pytest

from tests.gpu_util import build_kdom, ensure_built
from workload import configs, gpu_gen

pytestmark = pytest.mark.gpu

SHORT_NS = 2_000_000   # 2 ms: far above a clean step (tens of microseconds)


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    ensure_built()


# the two fused kernels: the single-exchange kernel at the 32K single-sequence
# shape (its whole first-round list resident) and at batch 8 (32 units,
# clusters of 4, the list streamed), the cluster kernel at batch 16 (64
# units, clusters of 2)
CASES = [("llama3_8b_ctx32k", {}, 1), ("qwen25_7b_b8_ctx16k", dict(context=4096), 1),
         ("qwen25_7b_b8_ctx16k", dict(context=4096, batch=16), 0)]


def _setup(name="llama3_8b_ctx32k", over=None, kernel=1):
    import torch
    from kv_cache_token_tip_gb300 import dims_for, fasa_step_kernel, fasa_workspace_size
    cfg = configs.CONFIGS[name].with_(**(over or {}))
    dims = dims_for(cfg)
    assert fasa_step_kernel(dims) == kernel
    L = gpu_gen.make_layer(cfg, 0)
    kd = build_kdom(L, dims)
    n = fasa_workspace_size(dims, cfg.budget)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda") if n else None
    return cfg, dims, L, kd, ws


def _step(cfg, dims, L, kd, ws):
    import torch
    from kv_cache_token_tip_gb300 import fasa_decode_step
    out = torch.full((cfg.batch, cfg.n_q_heads, cfg.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.full((cfg.batch, cfg.n_kv_heads, cfg.budget), -1, dtype=torch.int32, device="cuda")
    cnt = torch.full((cfg.batch, cfg.n_kv_heads), -1, dtype=torch.int32, device="cuda")
    fasa_decode_step(L.q, L.pos, L.k, L.v, kd, L.dom_fc, L.seq_lens, cfg.budget, out, idx, cnt, ws, dims)
    return out, idx, cnt


@pytest.mark.parametrize("name,over,kernel", CASES)
def test_short_wait_bound_alone_changes_nothing(name, over, kernel):
    from kv_cache_token_tip_gb300 import fasa_device_status, fasa_test_fault_injection
    cfg, dims, L, kd, ws = _setup(name, over, kernel)
    fasa_device_status()
    out0, idx0, cnt0 = _step(cfg, dims, L, kd, ws)
    assert fasa_device_status() == 0
    try:
        fasa_test_fault_injection(wait_limit_ns=SHORT_NS)
        out1, idx1, cnt1 = _step(cfg, dims, L, kd, ws)
        st = fasa_device_status()
    finally:
        fasa_test_fault_injection()
    assert st == 0
    assert np.array_equal(idx1.cpu().numpy(), idx0.cpu().numpy())
    assert np.array_equal(cnt1.cpu().numpy(), cnt0.cpu().numpy())
    assert np.array_equal(out1.cpu().numpy(), out0.cpu().numpy())


@pytest.mark.parametrize("name,over,kernel", CASES)
def test_unissued_tip_copy_times_out_and_the_stream_stays_usable(name, over, kernel):
    import torch
    from kv_cache_token_tip_gb300 import FASA_DEV_TIMEOUT, fasa_device_status, fasa_test_fault_injection
    cfg, dims, L, kd, ws = _setup(name, over, kernel)
    fasa_device_status()
    out0, idx0, cnt0 = _step(cfg, dims, L, kd, ws)
    assert fasa_device_status() == 0
    try:
        fasa_test_fault_injection(wait_limit_ns=SHORT_NS, drop_tip_tile=0)
        t0 = time.perf_counter()
        _step(cfg, dims, L, kd, ws)
        st = fasa_device_status()          # synchronises the stream
        elapsed = time.perf_counter() - t0
    finally:
        fasa_test_fault_injection()
    assert st & FASA_DEV_TIMEOUT, f"status {st}"
    # the copy wait, the drain and the peer exchanges are each bounded:
    # the launch ends within a small multiple of the bound
    assert elapsed < 2.0, f"faulted step took {elapsed:.3f} s"
    # the context and the stream still work, and the next clean step is
    # unaffected by the barrier state the faulted one left behind
    out2, idx2, cnt2 = _step(cfg, dims, L, kd, ws)
    assert fasa_device_status() == 0
    torch.cuda.synchronize()
    assert np.array_equal(idx2.cpu().numpy(), idx0.cpu().numpy())
    assert np.array_equal(cnt2.cpu().numpy(), cnt0.cpu().numpy())
    assert np.array_equal(out2.cpu().numpy(), out0.cpu().numpy())


def test_withheld_fac_refill_times_out_and_the_stream_stays_usable():
    """The single-exchange kernel's FAC after the selection (batch 8,
    clusters of 4): when the warp that refills attending warp 0's slots
    withholds the completion report of one refill, warp 0's wait on that
    slot runs out within the bound (and the later waits of that warp, one
    phase behind, each within the bound too); FASA_DEV_TIMEOUT is reported,
    the launch ends, and the next clean step matches the one before it bit
    for bit.  The copies themselves are issued and land: nothing is left in
    flight."""
    import torch
    from kv_cache_token_tip_gb300 import FASA_DEV_TIMEOUT, fasa_device_status, fasa_test_fault_injection
    cfg, dims, L, kd, ws = _setup("qwen25_7b_b8_ctx16k", dict(context=4096), 1)
    fasa_device_status()
    out0, idx0, cnt0 = _step(cfg, dims, L, kd, ws)
    assert fasa_device_status() == 0
    try:
        fasa_test_fault_injection(wait_limit_ns=SHORT_NS, drop_fac_refill=0)
        t0 = time.perf_counter()
        _step(cfg, dims, L, kd, ws)
        st = fasa_device_status()
        elapsed = time.perf_counter() - t0
    finally:
        fasa_test_fault_injection()
    assert st & FASA_DEV_TIMEOUT, f"status {st}"
    assert elapsed < 2.0, f"faulted step took {elapsed:.3f} s"
    out2, idx2, cnt2 = _step(cfg, dims, L, kd, ws)
    assert fasa_device_status() == 0
    torch.cuda.synchronize()
    assert np.array_equal(idx2.cpu().numpy(), idx0.cpu().numpy())
    assert np.array_equal(cnt2.cpu().numpy(), cnt0.cpu().numpy())
    assert np.array_equal(out2.cpu().numpy(), out0.cpu().numpy())
