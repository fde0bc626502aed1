"""Benchmark of the FASA decode step on GB300.

One step = one fused decode step (RoPE(q) -> TIP -> top-k -> FAC) over one
batch of the named workload, launched through the C ABI.  Inputs are
synthetic (seeded) and resident in HBM; each step reads a different replica
so that the replicas together exceed the L2 cache several times over.

Prints ONE JSON line.  `value` is the achieved HBM throughput in TB/s of the
algorithmic bytes (K_dom columns of the cached tokens + selected K/V rows +
query + output), summed over ranks and divided by the slowest rank's time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fasa|reference]
                    [--workload NAME]

`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload (the reference arm of this path).
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workload import configs, synth  # noqa: E402

METRIC = "FASA decode-step µs and achieved HBM TB/s (TIP+top-k+FAC) at 32K ctx"
DEFAULT_WORKLOAD = "llama3_8b_ctx32k"
L2_BYTES = 129 * 1024 * 1024
TRIAL_S = 2.0  # target length of one timed trial when --steps is not given
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["kv_cache_token_tip_gb300/csrc/fasa_step.cuh",
                  "kv_cache_token_tip_gb300/csrc/fasa_cluster.cuh",
                  "kv_cache_token_tip_gb300/csrc/fasa_ptx.cuh",
                  "kv_cache_token_tip_gb300/csrc/fasa_internal.h",
                  "kv_cache_token_tip_gb300/csrc/fasa_api.cu"]
CA_SOURCES = ["kv_cache_token_tip_gb300/csrc/fasa_ca.cu",
              "kv_cache_token_tip_gb300/csrc/fasa_ptx.cuh"]
CA_METRIC = "FC calibration (Contextual Agreement of every FC): achieved HBM TB/s of the K cache read once"


# ----------------------------------------------------------------------------
# Byte model (FASA-C memory movement, per step)
# ----------------------------------------------------------------------------
def algorithmic_bytes(cfg, lens, budget=None) -> dict:
    """Bytes one layer's decode step must move: every cached token's
    dominant-FC key columns (TIP; each head its own count of FCs), the
    selected K and V rows (FAC), the query, the fp32 output and the small
    index tables."""
    es = cfg.elem_bytes
    H, d = cfg.n_kv_heads, cfg.head_dim
    n_sum = sum(cfg.head_n_tip(h) for h in range(H))
    budget = cfg.budget if budget is None else budget
    lens = np.asarray(lens, dtype=np.int64)
    tip = int(np.sum(lens) * n_sum * 2 * es)
    sel = int(np.sum(np.minimum(lens, budget)) * H * 2 * d * es)
    q = cfg.batch * cfg.n_q_heads * d * es
    out = cfg.batch * cfg.n_q_heads * d * 4
    small = H * cfg.n_tip * 4 + 2 * cfg.batch * 4   # the dominant-FC table and the lengths
    dense = int(np.sum(lens) * H * 2 * d * es) + q + out + 2 * cfg.batch * 4
    return dict(tip=tip, fac=sel, q=q, out=out, small=small,
                total=tip + sel + q + out + small, dense_total=dense)


def fasa_m_eq10_bytes(cfg) -> int:
    """Eq. 10 ("Hardware-Aware Variants", FASA-M) for one layer of the
    workload: per (batch, KV head), the dominant key columns of every cache
    slot (L = T_max, d_dom = 2 n_tip) plus the budget's worth of the other key
    dimensions and of values (b = the budget)."""
    d, es, d_dom = cfg.head_dim, cfg.elem_bytes, 2 * cfg.n_tip
    per_head = cfg.context * d_dom + cfg.budget * (d - d_dom) + cfg.budget * d
    return int(cfg.batch * cfg.n_kv_heads * per_head * es)


def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for f in (KERNEL_SOURCES if sources is None else sources):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic(workload: str, prefix: str = "fasa_step", sources=None):
    """DRAM bytes per launch (per call, for a call of several launches) from
    the committed ncu summary, if it was taken on the current kernel sources
    (else None)."""
    path = os.path.join(ROOT, "profiles", f"{prefix}_{workload}.md")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(sources)
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_hash") != want:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------
# Clock sampling during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------------------------
# Distributed plumbing (one process per GPU, independent replicas)
# ----------------------------------------------------------------------------
def dist_setup(n_gpus: int):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}")
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("FASA_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return rank, world, local, pg


def barrier(pg, device=None):
    if pg is not None:
        if device is not None and pg.get_backend() == "nccl":
            pg.barrier(device_ids=[device])
        else:
            pg.barrier()


def max_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    import torch
    dev = "cuda" if pg.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# CPU oracle leg (bounded sample)
# ----------------------------------------------------------------------------
def unit_bytes(cfg, L: int, h: int = 0) -> int:
    """Algorithmic bytes of one (batch, KV head h) unit of length L."""
    es, G, d = cfg.elem_bytes, cfg.group, cfg.head_dim
    return L * cfg.head_n_tip(h) * 2 * es + min(L, cfg.budget) * 2 * d * es + G * d * es + G * d * 4


def _wait_go(go):
    """Blocks until the parent process says go (a line on stdin), when asked."""
    if go:
        print("ready", flush=True)
        sys.stdin.readline()


def oracle_sample(cfg, seconds: float = 12.0, max_steps: int = 10 ** 9, warmup: int = 0, n_units: int = 2,
                  unit_offset: int = 0, go: bool = False):
    """Times the fp64 oracle (as it stands, single-threaded numpy) on a bounded
    sample of the workload: each step is one (batch, KV head) unit of the
    decode step -- RoPE of its query group, TIP over its cached tokens, TopK-I
    and FAC -- cycling over `n_units` units from `unit_offset`, host-generated
    with the workload's recipe.  Runs `warmup` untimed steps, then timed steps
    until `max_steps` or `seconds` is reached.  Returns (seconds, steps, bytes)."""
    import oracle as O
    lens = synth.seq_lens(cfg)
    G = cfg.group
    q_all = O.decode_stored(synth.store(synth.gen_q(cfg, 0), cfg.dtype), cfg.dtype)
    dom = synth.dominant_fcs(cfg, 0)
    units = []
    n_all = cfg.batch * cfg.n_kv_heads
    for uu in range(min(n_units, n_all)):
        u = (unit_offset + uu) % n_all
        b, h = divmod(u, cfg.n_kv_heads)
        L = int(lens[b])
        kk, vv = synth.gen_kv_head(cfg, 0, b, h, t_count=L)
        K = O.decode_stored(synth.store(kk, cfg.dtype), cfg.dtype)
        V = O.decode_stored(synth.store(vv, cfg.dtype), cfg.dtype)
        units.append((q_all[b, h * G:(h + 1) * G], int(lens[b]), K, V, O.dominant_set(dom[h]),
                      unit_bytes(cfg, L, h)))

    def one(i):
        q, pos, K, V, dfc, nb = units[i % len(units)]
        q_rot = O.apply_rope_q(q[None], np.array([pos]), cfg.rope_theta)[0]
        s = O.tip_scores_unit(q_rot, K, dfc)
        idx = O.topk_select_unit(s, cfg.budget)
        O.focused_attention_unit(q_rot, K, V, idx)
        return nb

    warm_until = time.perf_counter() + min(5.0, seconds)
    for i in range(warmup):   # untimed; bounded in time like the timed part
        one(i)
        if time.perf_counter() >= warm_until:
            break
    _wait_go(go)
    steps, nbytes = 0, 0
    t0 = time.perf_counter()
    while steps < max_steps:
        nbytes += one(steps)
        steps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return time.perf_counter() - t0, steps, nbytes


def oracle_ca_sample(cfg, seconds: float = 12.0, max_steps: int = 10 ** 9, warmup: int = 0, n_units: int = 1,
                     unit_offset: int = 0, go: bool = False):
    """Times the fp64 oracle's calibration on a bounded sample: each step is one
    (batch, KV head) unit -- RoPE of its query group at position len, then the
    Contextual Agreement (Eq. 4) of every FC over its cached tokens with K = the
    workload's budget.  Returns (seconds, steps, bytes of K read once)."""
    import oracle as O
    lens = synth.seq_lens(cfg)
    G = cfg.group
    q_all = O.decode_stored(synth.store(synth.gen_q(cfg, 0), cfg.dtype), cfg.dtype)
    units = []
    n_all = cfg.batch * cfg.n_kv_heads
    for uu in range(min(n_units, n_all)):
        u = (unit_offset + uu) % n_all
        b, h = divmod(u, cfg.n_kv_heads)
        L = int(lens[b])
        kk, _ = synth.gen_kv_head(cfg, 0, b, h, t_count=L)
        K = O.decode_stored(synth.store(kk, cfg.dtype), cfg.dtype)
        units.append((q_all[b, h * G:(h + 1) * G], L, K, L * cfg.head_dim * cfg.elem_bytes))

    def one(i):
        q, pos, K, nb = units[i % len(units)]
        q_rot = O.apply_rope_q(q[None], np.array([pos]), cfg.rope_theta)[0]
        O.contextual_agreement_unit(q_rot, K, cfg.budget)
        return nb

    warm_until = time.perf_counter() + min(5.0, seconds)
    for i in range(warmup):   # untimed; bounded in time like the timed part
        one(i)
        if time.perf_counter() >= warm_until:
            break
    _wait_go(go)
    steps, nbytes = 0, 0
    t0 = time.perf_counter()
    while steps < max_steps:
        nbytes += one(steps)
        steps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return time.perf_counter() - t0, steps, nbytes


def run_oracle_leg(cfg, seconds: float, max_steps: int = 10 ** 9, warmup: int = 0, fn: str = "oracle_sample",
                   procs: int = 0):
    """Runs oracle_sample (or `fn`) on every host core: one child process per
    core, each with BLAS limited to one thread and its own units of the
    workload.  The children set up their inputs, then start their timed loops
    together; the result sums their steps and bytes over the longest timed
    loop.  Returns dict(seconds, steps, bytes, procs, steps_per_proc)."""
    procs = procs or (os.cpu_count() or 1)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    kids = []
    for i in range(procs):
        code = ("import json,sys; sys.path.insert(0, %r); import bench; from workload import configs; "
                "cfg = configs.CONFIGS[%r]; t, n, b = bench.%s(cfg, %r, %r, %r, unit_offset=%d, go=True); "
                "print(json.dumps({'seconds': t, 'steps': n, 'bytes': b}), flush=True)"
                % (ROOT, cfg.name, fn, seconds, max_steps, warmup, 2 * i))
        kids.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdin=subprocess.PIPE,
                                     stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    try:
        for k in kids:   # every child has its inputs ready
            line = k.stdout.readline()
            if line.strip() != "ready":
                raise RuntimeError(f"oracle child failed before timing: {line!r} {k.stderr.read()[-2000:]}")
        for k in kids:
            k.stdin.write("go\n")
            k.stdin.flush()
        res = []
        for k in kids:
            out, err = k.communicate(timeout=1800)
            if k.returncode != 0:
                raise RuntimeError(err[-2000:])
            res.append(json.loads(out.strip().splitlines()[-1]))
    finally:
        for k in kids:
            if k.poll() is None:
                k.kill()
    return dict(seconds=max(r["seconds"] for r in res), steps=sum(r["steps"] for r in res),
                bytes=sum(r["bytes"] for r in res), procs=procs,
                steps_per_proc=max(r["steps"] for r in res))


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def make_replicas(cfg, R, dims):
    import torch
    from kv_cache_token_tip_gb300 import fasa_build_kdom
    from workload import gpu_gen
    reps = []
    for r in range(R):
        L = gpu_gen.make_layer(cfg, layer=r)
        kd = torch.empty((cfg.batch, cfg.n_kv_heads, cfg.context // 64, cfg.n_tip, 64, 2), dtype=L.k.dtype,
                         device="cuda")
        fasa_build_kdom(L.k, L.dom_fc, L.seq_lens, kd, dims)
        reps.append((L, kd))
    torch.cuda.synchronize()
    return reps


SUBMIT_DELAY_S = 100e-6


def gpu_delay(seconds: float):
    """A bounded spin on the GPU (torch's sleep kernel, about `seconds` at the
    maximum SM clock) on the current stream."""
    import torch
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        sleep(int(seconds * 2.07e9))


def capture(fn, n_steps, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_steps):
                fn(i)
    return g


def run_gpu(args):
    import torch
    from kv_cache_token_tip_gb300 import build as kbuild
    kbuild.build()
    from kv_cache_token_tip_gb300 import (FASA_KERNEL_SINGLE_EXCHANGE, dims_for, fasa_apply_rope_q,
                                          fasa_cluster_size, fasa_decode_step, fasa_decode_step_split,
                                          fasa_dense_attention, fasa_device_status, fasa_step_kernel,
                                          fasa_workspace_size)

    rank, world, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    cfg = configs.CONFIGS[args.workload]
    dims = dims_for(cfg)
    lens = synth.seq_lens(cfg)
    layers = cfg.layers          # a decode step runs every layer: one launch each
    # the byte model summed over the layers (each layer its own budget)
    per_layer = [algorithmic_bytes(cfg, lens, cfg.layer_budget(l)) for l in range(layers)]
    model = {kk: sum(m[kk] for m in per_layer) / layers for kk in per_layer[0]}
    if args.append:  # the new token's K and V rows and K_dom entries are written
        model["append"] = cfg.batch * sum(2 * cfg.head_dim + 2 * cfg.head_n_tip(h)
                                          for h in range(cfg.n_kv_heads)) * cfg.elem_bytes
        model["total"] += model["append"]
    per_step = int(round(model["total"] * layers))
    if layers > 1:
        R = layers               # one replica per layer, launched in order
    else:
        R = max(4, int(np.ceil(4 * L2_BYTES / per_step)))
        R = min(R, 64)
    if args.replicas > 0:  # profiling runs only: fewer replicas may fit in L2
        R = args.replicas
    reps = make_replicas(cfg, R, dims)
    split = args.fasa_m and not args.append
    if args.fasa_m:
        # FASA-M placement ("Hardware-Aware Variants"): the values and the
        # keys' non-dominant FC pairs (K^nondom) in page-locked host memory,
        # the dominant key cache K_dom on the GPU.  The split step moves only
        # the selected rows' K^nondom and V over the host link and rebuilds
        # each key with its K_dom pairs.  (The dense comparison, and the
        # append step, read whole keys from host memory.)
        from kv_cache_token_tip_gb300 import fasa_build_knondom
        ndp = cfg.head_dim // 2 - cfg.n_tip
        for L, _ in reps:
            if split:
                L.knd = torch.empty((cfg.batch, cfg.n_kv_heads, cfg.context, 2 * ndp), dtype=L.k.dtype,
                                    pin_memory=True)
                fasa_build_knondom(L.k, L.dom_fc, None, L.knd, dims)
                torch.cuda.synchronize()
            L.k = L.k.cpu().pin_memory()
            L.v = L.v.cpu().pin_memory()
        torch.cuda.empty_cache()
        if fasa_device_status():
            raise RuntimeError("K^nondom build reported bad input")
    B, Hq, H, d, k = cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.budget
    ws_bytes = fasa_workspace_size(dims, k)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda") if ws_bytes else None
    outs = [torch.empty((B, Hq, d), dtype=torch.float32, device="cuda") for _ in range(R)]
    stream = torch.cuda.Stream()

    if args.append:
        # fasa_decode_step_append with lengths one short of the cache: each
        # step stores its token at index len - 1 (the same slot on every
        # replay) and attends over the same len tokens as the plain step
        from kv_cache_token_tip_gb300 import fasa_decode_step_append
        gen = torch.Generator(device="cuda").manual_seed(1)
        app = []
        for L, _ in reps:
            shape = (B, H, cfg.head_dim)
            kn = torch.randn(shape, generator=gen, device="cuda").to(L.k.dtype)
            vn = torch.randn(shape, generator=gen, device="cuda").to(L.v.dtype)
            app.append((kn, vn, (L.seq_lens - 1).contiguous()))

    def step(i):
        L, kd = reps[i % R]
        kl = cfg.layer_budget(i % layers)
        if args.append:
            kn, vn, lens_m1 = app[i % R]
            fasa_decode_step_append(L.q, kn, vn, lens_m1, L.k, L.v, kd, L.dom_fc, kl, outs[i % R],
                                    None, None, ws, dims, stream=stream)
        elif split:
            fasa_decode_step_split(L.q, L.pos, L.knd, L.v, kd, L.dom_fc, L.seq_lens, kl, outs[i % R],
                                   None, None, ws, dims, stream=stream)
        else:
            fasa_decode_step(L.q, L.pos, L.k, L.v, kd, L.dom_fc, L.seq_lens, kl, outs[i % R],
                             None, None, ws, dims, stream=stream)

    # dense comparison: the same kernels over every cached row
    q_rots = []
    for L, _ in reps:
        qr = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
        fasa_apply_rope_q(L.q, L.pos, qr, dims)
        q_rots.append(qr)

    def dense_step(i):
        L, _ = reps[i % R]
        fasa_dense_attention(q_rots[i % R], L.k, L.v, L.seq_lens, outs[i % R], dims, stream=stream)

    step(0)            # first calls outside capture: attribute set-up and caches
    dense_step(0)
    torch.cuda.synchronize()
    chunk = R * max(1, 512 // R)
    W = args.warmup if args.warmup is not None else max(8, 2048 // layers)
    g_chunk = capture(step, chunk, stream)
    g_warm = capture(step, W * layers, stream) if W else None
    torch.cuda.synchronize()
    # the warm-up, timed: without --steps, K is chosen so that one trial
    # lasts about TRIAL_S (the same K on every rank)
    wev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    with torch.cuda.stream(stream):
        wev[0].record(stream)
        (g_warm if g_warm is not None else g_chunk).replay()
        wev[1].record(stream)
    torch.cuda.synchronize()
    warm_launches = W * layers if g_warm is not None else chunk
    t_step = max_over_ranks(pg, wev[0].elapsed_time(wev[1])) / 1e3 / warm_launches * layers
    K = args.steps if args.steps else int(min(200000, max(20, round(TRIAL_S / t_step))))
    KL = K * layers              # timed launches
    rem = KL % chunk
    g_rem = capture(step, rem, stream) if rem else None
    torch.cuda.synchronize()
    status = fasa_device_status(stream)
    if status:
        raise RuntimeError(f"device status {status} after warm-up")

    # T trials of exactly K timed steps each; the reported time is the median
    # trial.  Before each trial a short GPU-side delay (a bounded spin) keeps
    # the GPU busy while the host submits the graphs, so the trial times
    # device execution, not graph submission.
    trials = max(1, args.trials)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(trials)]
    barrier(pg, local)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):   # graphs replay on the current stream
            for ev0, ev1 in evs:
                gpu_delay(SUBMIT_DELAY_S)
                ev0.record(stream)
                for _ in range(KL // chunk):
                    g_chunk.replay()
                if g_rem is not None:
                    g_rem.replay()
                ev1.record(stream)
        torch.cuda.synchronize()
    barrier(pg, local)
    torch.cuda.synchronize()
    trial_ms = [max_over_ranks(pg, ev0.elapsed_time(ev1)) for ev0, ev1 in evs]
    sec_per_step = statistics.median(trial_ms) / 1e3 / K

    # dense baseline (same machinery), fewer steps
    Kd = max(R, min(K // 8, 4096))
    g_dense = capture(dense_step, Kd, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g_dense.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        g_dense.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    dense_sec = e0.elapsed_time(e1) / 1e3 / Kd * layers   # per decode step

    # end to end through the public API: every step copies that step's q, pos
    # and lens from pinned host memory (one packed copy), runs
    # fasa_decode_step and copies the output back to pinned host memory, then
    # the host synchronises.  The three calls are captured once per replica in
    # a CUDA graph and replayed per step (graph mode); the same three calls
    # issued eagerly from Python are timed as well (eager mode).
    E = min(2000, max(50, K // 100))
    qbytes = reps[0][0].q.numel() * reps[0][0].q.element_size()
    qoff = (qbytes + 15) // 16 * 16
    nbytes = qoff + 2 * B * 4
    h_in = [torch.empty(nbytes, dtype=torch.uint8).pin_memory() for _ in range(R)]
    d_in = [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in range(R)]
    lens32 = torch.from_numpy(np.asarray(lens, dtype=np.int32))
    for r in range(R):
        h_in[r][:qbytes].copy_(reps[r][0].q.cpu().contiguous().view(torch.uint8).reshape(-1))
        h_in[r][qoff:qoff + 4 * B].copy_(lens32.view(torch.uint8))          # pos = len
        h_in[r][qoff + 4 * B:].copy_(lens32.view(torch.uint8))
    d_q = [d_in[r][:qbytes].view(reps[0][0].q.dtype).view(reps[0][0].q.shape) for r in range(R)]
    d_pos = [d_in[r][qoff:qoff + 4 * B].view(torch.int32) for r in range(R)]
    d_lens = [d_in[r][qoff + 4 * B:].view(torch.int32) for r in range(R)]
    h_out = [torch.empty((B, Hq, d), dtype=torch.float32).pin_memory() for _ in range(R)]

    def e2e_step(r):
        L, kd = reps[r]
        d_in[r].copy_(h_in[r], non_blocking=True)
        fasa_decode_step(d_q[r], d_pos[r], L.k, L.v, kd, L.dom_fc, d_lens[r], cfg.layer_budget(r % layers),
                         outs[r], None, None, ws, dims,
                         stream=stream)
        h_out[r].copy_(outs[r], non_blocking=True)

    with torch.cuda.stream(stream):
        for r in range(R):
            e2e_step(r)
    torch.cuda.synchronize()
    graphs = []
    for r in range(R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                e2e_step(r)
        graphs.append(g)
    torch.cuda.synchronize()
    barrier(pg, local)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(E):
            for l in range(layers):
                graphs[(i * layers + l) % R].replay()
            stream.synchronize()
    e2e_sec = max_over_ranks(pg, time.perf_counter() - t0)
    e2e_per_step = e2e_sec / E
    barrier(pg, local)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(E):
            for l in range(layers):
                e2e_step((i * layers + l) % R)
            stream.synchronize()
    e2e_eager_per_step = max_over_ranks(pg, time.perf_counter() - t0) / E
    last = ((E - 1) * layers + layers - 1) % R
    if not torch.equal(h_out[last], outs[last].cpu()):
        raise RuntimeError("end-to-end output copy does not match the device output")

    # zero-copy: the step reads q/pos/lens from the same pinned host buffers
    # and writes its output into pinned host memory in place (the library's
    # host-resident step I/O), so each step is one graph of one launch
    h_q = [h_in[r][:qbytes].view(reps[0][0].q.dtype).view(reps[0][0].q.shape) for r in range(R)]
    h_pos = [h_in[r][qoff:qoff + 4 * B].view(torch.int32) for r in range(R)]
    h_lens = [h_in[r][qoff + 4 * B:].view(torch.int32) for r in range(R)]
    h_out_zc = [torch.empty((B, Hq, d), dtype=torch.float32).pin_memory() for _ in range(R)]

    def zc_step(r):
        L, kd = reps[r]
        fasa_decode_step(h_q[r], h_pos[r], L.k, L.v, kd, L.dom_fc, h_lens[r], cfg.layer_budget(r % layers),
                         h_out_zc[r], None, None, ws, dims, stream=stream)

    with torch.cuda.stream(stream):
        for r in range(R):
            zc_step(r)
    torch.cuda.synchronize()
    zc_graphs = []
    for r in range(R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                zc_step(r)
        zc_graphs.append(g)
    torch.cuda.synchronize()
    barrier(pg, local)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(E):
            for l in range(layers):
                zc_graphs[(i * layers + l) % R].replay()
            stream.synchronize()
    zc_per_step = max_over_ranks(pg, time.perf_counter() - t0) / E
    if not torch.equal(h_out_zc[last], outs[last].cpu()):
        raise RuntimeError("zero-copy output does not match the device output")
    status = fasa_device_status(stream)
    if status:
        raise RuntimeError(f"device status {status} after the timed region")

    peak, peak_kind = measured_peak()
    achieved_gbs = per_step / sec_per_step / 1e9
    clocks = clk.summary()
    C = fasa_cluster_size(dims)
    kernel_name = (f"fasa_step_kernel<{cfg.head_dim}>" if fasa_step_kernel(dims) == FASA_KERNEL_SINGLE_EXCHANGE
                   else f"fasa_cluster_kernel<{cfg.dtype},{cfg.head_dim}>")
    line = None
    if args.cpu_baseline and rank == 0 and world == 1:
        cb = run_oracle_leg(cfg, args.cpu_seconds)
        cpu = {"value": cb["bytes"] / cb["seconds"] / 1e12, "unit": "TB/s", "cores": cb["procs"], "kind": "oracle",
               "sample": f"{cb['steps']} (batch, KV head) units of {cfg.name} in {cb['seconds']:.1f} s on "
                         f"{cb['procs']} host cores (one process per core, 1 BLAS thread each, timed loops "
                         f"started together; host-generated inputs, numpy fp64); "
                         f"{cb['seconds'] / cb['steps'] * B * H * layers * 1e6:.0f} us per whole decode step"}
    else:
        cpu = None
    if rank == 0:
        h2d = int(nbytes) * layers
        d2h = int(h_out[0].numel() * 4) * layers
        line = {
            "metric": METRIC,
            "value": round(world * per_step / sec_per_step / 1e12, 4),
            "unit": "TB/s",
            "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": round(sec_per_step * 1e3, 6),
            "us_per_step": round(sec_per_step * 1e6, 3),
            "trials": {"n": trials, "statistic": "median",
                       "us_per_step": [round(t * 1e3 / K, 3) for t in trial_ms],
                       "timing": f"{trials} trials of exactly {K} steps (CUDA-graph replay, CUDA events on the "
                                 f"launching stream; a {SUBMIT_DELAY_S * 1e6:.0f} us GPU spin before each trial "
                                 f"keeps graph submission out of the timed region)"},
            "tokens_per_s": round(world * B / sec_per_step, 1),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": cfg.dtype,
            "data": "synthetic (seeded; pre-RoPE q/k ~ N(0,1) with x8 outlier FCs, v ~ N(0,1))",
            "config": {"workload": cfg.name, "batch": B, "q_heads": Hq, "kv_heads": H, "head_dim": d,
                       "context": cfg.context, "n_tip": cfg.n_tip, "budget": k, "rope_theta": cfg.rope_theta,
                       **({"n_tip_per_head": list(cfg.n_tip_per_head)} if cfg.n_tip_per_head else {}),
                       **({"budget_per_layer": f"{cfg.budget_per_layer[0]} .. {cfg.budget_per_layer[-1]} "
                                               f"(mean {np.mean(cfg.budget_per_layer):.0f})"}
                          if cfg.budget_per_layer else {}),
                       "cluster_ctas": C, "replicas": R,
                       "l2": f"{'inputs larger than L2' if R * per_step > L2_BYTES else 'NOT larger than L2 (profiling run)'}: "
                             f"{R} replicas x {per_step / 1e6:.2f} MB/step "
                             f"rotate ({R * per_step / L2_BYTES:.1f}x L2)",
                       "launch": ("CUDA graph of fasa_decode_step launches, one kernel per step"
                                  if layers == 1 else
                                  f"CUDA graph of fasa_decode_step launches, one kernel per layer, "
                                  f"{layers} layers per step"),
                       "layers": layers,
                       "entry": "fasa_decode_step_append (each step stores its own token)" if args.append
                                else "fasa_decode_step",
                       "kv_placement": ("FASA-M split keys: K^nondom and V in pinned host memory, K_dom on "
                                        "the GPU; the selected rows' K^nondom and V cross the host link"
                                        if split else
                                        "pinned host memory (FASA-M): selected rows cross the host link"
                                        if args.fasa_m else "device memory"),
                       "parallelism": f"replicas x{world}"},
            "bytes_per_step": per_step,
            **({"fasa_m": {"key_layout": "split" if split else "whole keys",
                           # per selected row: d - 2 N_tip key elements and d value
                           # elements over the link (whole keys: 2 d)
                           "link_bytes_per_step": int(round(model["fac"] * layers * (
                               (2 * cfg.head_dim - 2 * cfg.n_tip) / (2 * cfg.head_dim) if split else 1.0))),
                           "link_bytes_whole_keys": int(round(model["fac"] * layers)),
                           "pages_formula_bytes": int(cfg.batch * cfg.n_kv_heads * cfg.budget
                                                      * (2 * cfg.head_dim - 2 * cfg.n_tip) * cfg.elem_bytes),
                           "link_gbs": round(model["fac"] * layers * (
                               (2 * cfg.head_dim - 2 * cfg.n_tip) / (2 * cfg.head_dim) if split else 1.0)
                               / sec_per_step / 1e9, 1),
                           "hbm_bytes_not_held_per_replica": int(2 * reps[0][0].k.numel()
                                                                 * reps[0][0].k.element_size()),
                           # what one layer's step keeps in HBM (the library allocates
                           # nothing), against Eq. 10's estimate for the layer
                           "hbm_bytes_held_per_replica": int(sum(
                               t.numel() * t.element_size() for t in (reps[0][1], reps[0][0].q, reps[0][0].pos,
                                                                      reps[0][0].seq_lens, reps[0][0].dom_fc,
                                                                      outs[0]))),
                           "workspace_bytes": int(ws.numel()) if ws is not None else 0,
                           "eq10_bytes_per_replica": fasa_m_eq10_bytes(cfg)}}
               if args.fasa_m else {}),
            "bytes_breakdown": {kk: int(round(model[kk] * layers))
                                for kk in ("tip", "fac", "q", "out", "small", "append")
                                if kk in model},
            "roofline": {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved_gbs / peak, 4),
                         # (the committed captures are of the plain step with the caches in device
                         # memory: no figure for the split-key or append forms)
                         "traffic": None if (args.fasa_m or args.append) else ncu_traffic(cfg.name),
                         "peak_kind": peak_kind, "kernel": kernel_name},
            "dense": {"us_per_step": round(dense_sec * 1e6, 3),
                      "achieved_gbs": round(model["dense_total"] * layers / dense_sec / 1e9, 1),
                      "sparse_vs_dense_speedup": round(dense_sec / sec_per_step, 3)},
            "e2e": {"value": round(world * per_step / zc_per_step / 1e12, 4), "unit": "TB/s",
                    "us_per_step": round(zc_per_step * 1e6, 3),
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "mode": "zero-copy: fasa_decode_step reads q/pos/lens from pinned host memory and writes out "
                            "into pinned host memory in place (one CUDA graph of one launch per step); host sync "
                            "every step",
                    "copy_us_per_step": round(e2e_per_step * 1e6, 3),
                    "copy_mode": "CUDA graph per step: pinned H2D copy of q/pos/lens, fasa_decode_step, D2H copy "
                                 "of out; host sync every step",
                    "copy_eager_us_per_step": round(e2e_eager_per_step * 1e6, 3)},
            "gpu_launches": K * layers,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return line


def run_calibrate(args):
    """The offline calibration (fasa_fc_agreement: the Contextual Agreement of
    every FC for every (batch, KV head) of the workload, K = its budget), timed
    like the decode step: CUDA graphs of calls rotating over input replicas
    that together exceed L2, W warm-up calls, then exactly K timed calls."""
    import torch
    from kv_cache_token_tip_gb300 import build as kbuild
    kbuild.build()
    from kv_cache_token_tip_gb300 import (dims_for, fasa_apply_rope_q, fasa_device_status, fasa_fc_agreement,
                                          fasa_fc_agreement_workspace_size)
    from workload import gpu_gen

    rank, world, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    cfg = configs.CONFIGS[args.workload]
    dims = dims_for(cfg)
    lens = synth.seq_lens(cfg)
    B, Hq, H, d = cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    k_bytes = int(np.sum(lens)) * H * d * cfg.elem_bytes          # the K cache, read once
    io_bytes = B * Hq * d * 4 + B * 4 + B * H * (d // 2) * 4       # q_rot, lengths, ca
    per_call = k_bytes + io_bytes
    R = args.replicas if args.replicas > 0 else min(16, max(2, int(np.ceil(4 * L2_BYTES / k_bytes))))
    reps = []
    for r in range(R):
        L = gpu_gen.make_layer(cfg, layer=r)
        L.v = None
        qr = torch.empty((B, Hq, d), dtype=torch.float32, device="cuda")
        fasa_apply_rope_q(L.q, L.pos, qr, dims)
        reps.append((L, qr, torch.empty((B, H, d // 2), dtype=torch.float32, device="cuda")))
    torch.cuda.empty_cache()
    ws = torch.empty(fasa_fc_agreement_workspace_size(dims), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()

    def call(i):
        L, qr, ca = reps[i % R]
        fasa_fc_agreement(qr, L.k, L.seq_lens, cfg.budget, ca, dims, workspace=ws, stream=stream)

    call(0)
    torch.cuda.synchronize()
    K, W = (args.steps or 2000), (args.warmup if args.warmup is not None else 64)
    chunk = R * max(1, 64 // R)
    g_chunk = capture(call, chunk, stream)
    rem = K % chunk
    g_rem = capture(call, rem, stream) if rem else None
    g_warm = capture(call, W, stream)
    with torch.cuda.stream(stream):
        g_warm.replay()
    torch.cuda.synchronize()
    if fasa_device_status(stream):
        raise RuntimeError("device status set after warm-up")
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg, local)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(K // chunk):
                g_chunk.replay()
            if g_rem is not None:
                g_rem.replay()
            ev1.record(stream)
        torch.cuda.synchronize()
    barrier(pg, local)
    torch.cuda.synchronize()
    sec = max_over_ranks(pg, ev0.elapsed_time(ev1)) / 1e3 / K

    # end to end through the public API: per call, a pinned H2D copy of the
    # rotated queries and lengths (the K cache is resident model state), the
    # call, a D2H copy of ca, a host sync
    E = max(20, min(500, K))
    qb = reps[0][1].numel() * 4
    h_in = torch.empty(qb + 4 * B, dtype=torch.uint8).pin_memory()
    h_in[:qb].copy_(reps[0][1].cpu().view(torch.uint8).reshape(-1))
    h_in[qb:].copy_(torch.from_numpy(np.asarray(lens, dtype=np.int32)).view(torch.uint8))
    d_in = torch.empty_like(h_in, device="cuda")
    d_q = d_in[:qb].view(torch.float32).view(B, Hq, d)
    d_len = d_in[qb:].view(torch.int32)
    h_out = torch.empty((B, H, d // 2), dtype=torch.float32).pin_memory()
    L0, _, ca0 = reps[0]

    def e2e():
        d_in.copy_(h_in, non_blocking=True)
        fasa_fc_agreement(d_q, L0.k, d_len, cfg.budget, ca0, dims, workspace=ws, stream=stream)
        h_out.copy_(ca0, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            e2e()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(E):
            g.replay()
            stream.synchronize()
    e2e_sec = max_over_ranks(pg, time.perf_counter() - t0) / E
    if not torch.equal(h_out, ca0.cpu()):
        raise RuntimeError("end-to-end output copy does not match the device output")
    if fasa_device_status(stream):
        raise RuntimeError("device status set after the timed region")

    peak, peak_kind = measured_peak()
    achieved = per_call / sec / 1e9
    line = None
    cpu = None
    if args.cpu_baseline and rank == 0 and world == 1:
        cb = run_oracle_leg(cfg, args.cpu_seconds, fn="oracle_ca_sample")
        cpu = {"value": cb["bytes"] / cb["seconds"] / 1e12, "unit": "TB/s", "cores": cb["procs"], "kind": "oracle",
               "sample": f"{cb['steps']} (batch, KV head) units of {cfg.name} in {cb['seconds']:.1f} s on "
                         f"{cb['procs']} host cores (one process per core, 1 BLAS thread each; host-generated "
                         f"inputs, numpy fp64); "
                         f"{cb['seconds'] / cb['steps'] * B * H * 1e3:.0f} ms per whole call"}
    if rank == 0:
        line = {
            "metric": CA_METRIC,
            "value": round(world * per_call / sec / 1e12, 4), "unit": "TB/s",
            "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": round(sec * 1e3, 6), "us_per_step": round(sec * 1e6, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic (seeded; pre-RoPE q/k ~ N(0,1) with x8 outlier FCs)",
            "config": {"workload": cfg.name, "batch": B, "q_heads": Hq, "kv_heads": H, "head_dim": d,
                       "context": cfg.context, "topk": cfg.budget, "replicas": R,
                       "l2": f"{'inputs larger than L2' if R * k_bytes > L2_BYTES else 'NOT larger than L2'}: "
                             f"{R} replicas x {k_bytes / 1e6:.1f} MB of K rotate",
                       "entry": "fasa_fc_agreement (3 launches: scores, per-row TopK-I masks, per-FC counts)",
                       "parallelism": f"replicas x{world}"},
            "bytes_per_step": per_call,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": ncu_traffic(cfg.name, "fasa_ca", CA_SOURCES),
                         "peak_kind": peak_kind, "kernel": "fasa_fc_agreement (all 3 launches of one call)"},
            "e2e": {"value": round(world * per_call / e2e_sec / 1e12, 4), "unit": "TB/s",
                    "us_per_step": round(e2e_sec * 1e6, 3), "h2d_bytes_per_step": int(h_in.numel()),
                    "d2h_bytes_per_step": int(h_out.numel() * 4),
                    "mode": "CUDA graph per call: pinned H2D of q_rot/lens, fasa_fc_agreement, D2H of ca"},
            "gpu_launches": 3 * K,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return line


def run_reference(args):
    """The reference arm: the fp64 oracle timed on every host core.  One step
    is one (batch, KV head) unit of the workload on each core at once (a
    bounded sample); W untimed warm-up steps, then at most K timed steps,
    stopped after --cpu-seconds."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return None
    cfg = configs.CONFIGS[args.workload]
    cal = args.calibrate
    warm = args.warmup if args.warmup is not None else 3
    cb = run_oracle_leg(cfg, args.cpu_seconds, args.steps or 10 ** 9, warm,
                        fn="oracle_ca_sample" if cal else "oracle_sample")
    val = cb["bytes"] / cb["seconds"] / 1e12
    per_step = cb["seconds"] / cb["steps_per_proc"]
    line = {
        "impl": "reference",
        "metric": CA_METRIC if cal else METRIC, "value": val, "unit": "TB/s", "n_gpus": world,
        "steps": cb["steps_per_proc"], "warmup": warm,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, host-generated)",
        "config": {"workload": cfg.name, "batch": cfg.batch, "q_heads": cfg.n_q_heads,
                   "kv_heads": cfg.n_kv_heads, "head_dim": cfg.head_dim, "context": cfg.context,
                   "n_tip": cfg.n_tip, "budget": cfg.budget,
                   "step": f"one (batch, KV head) unit of the "
                           + ("calibration (CA of every FC, topk = budget)" if cal else "decode step")
                           + f" on each of {cb['procs']} host cores"},
        "cpu_baseline": {"value": val, "unit": "TB/s", "cores": cb["procs"], "kind": "oracle",
                         "sample": f"{cb['steps']} units in {cb['seconds']:.1f} s on {cb['procs']} cores, bounded "
                                   f"to ~{args.cpu_seconds:.0f} s (numpy fp64, one process per core, 1 BLAS "
                                   f"thread each)"},
        "e2e": {"value": val, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps per trial (default: as many as fill about %.0f s, at most 200000)" % TRIAL_S)
    ap.add_argument("--warmup", type=int, default=None,
                    help="untimed warm-up steps (default: 2048 launches' worth, at least 8 steps)")
    ap.add_argument("--impl", choices=["fasa", "reference"], default="fasa")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(configs.CONFIGS))
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--fasa-m", dest="fasa_m", action="store_true",
                    help="FASA-M placement: K/V caches in pinned host memory, K_dom on the GPU")
    ap.add_argument("--append", action="store_true",
                    help="time fasa_decode_step_append (the step stores its own token first) instead of "
                         "fasa_decode_step")
    ap.add_argument("--calibrate", action="store_true",
                    help="time the offline calibration (fasa_fc_agreement) instead of the decode step")
    ap.add_argument("--trials", type=int, default=5,
                    help="timed trials of K steps each; the median trial is reported")
    ap.add_argument("--replicas", type=int, default=0,
                    help="input replicas rotated through (0: enough to exceed 4x L2, as timing requires; "
                         "a smaller count is for profiler captures)")
    args = ap.parse_args(argv)
    if args.warmup is not None and args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.calibrate:
        return run_calibrate(args)
    return run_gpu(args)


if __name__ == "__main__":
    main()
