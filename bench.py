#!/usr/bin/env python
"""Benchmark of the INT8 KV cache decode step on GB300.

One step = the whole hot path over one batch of synthetic input: append one
new token (fp16 -> int8 codes + fp16 scales, written through the page table)
and split-K GQA decode attention over the dequantized cache with the per-head
combine.  Workload: batch 1, 16 query heads, 2 kv heads, head_dim 256, one
fp16 scale per 64 values, context 8192 (8191 cached + the appended token),
k8v8 store, K with 4 outlier channels per kv head (x20).

Inputs are resident in HBM when the timed region starts.  The pool is
replicated into enough copies (each step uses the next copy) that the bytes a
step reads were not left in L2 by the previous steps.  Steps are replayed
from a CUDA graph and timed with CUDA events on the launching stream.

Lines printed (rank 0, one JSON object):
  default            this library; ``value`` = algorithmic bytes per step /
                     device time per step (GB/s), plus ``e2e`` (the same metric
                     through the public API with pinned host buffers copied in
                     and the result copied out every step), ``roofline`` of the
                     decode kernel, ``cpu_baseline`` (the oracle on this host),
                     and ``extra`` (128K-context decode, k8v8 and k8v16).
  --impl reference   the oracle timed on the host cores on a bounded sample
                     of the same workload.
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("INT8-KV decode attn: achieved HBM GB/s (% of ~8 TB/s), μs/step at "
          "8K–128K ctx")
WORKLOAD = ("decode step (1-token append fused into the split-K GQA decode kernel, then the combine kernel): "
            "batch 1, 16 q heads, "
            "2 kv heads, head_dim 256, fp16 scale per 64 values, ctx 8192, k8v8, outlier K "
            "channels")

B, H, HKV, D, GS, PS, CTX = 1, 16, 2, 256, 64, 64, 8192


def step_bytes(ctx=CTX, hkv=HKV, h=H, d=D, gs=GS, k_int8=True, v_int8=True, append=True,
               v_q4=False, k_q4=False):
    """Algorithmic bytes of one step: int8 KV + scales (fp16 for an fp16 store;
    4-bit codes + one fp16 scale per 32 values for a 4-bit store) read once,
    q (fp16) read, O (fp32) written, and the appended token (fp16 in, codes +
    scales out)."""
    per_pos = 0
    for is8, is4 in ((k_int8, k_q4), (v_int8, v_q4)):
        if is4:
            per_pos += hkv * d // 2 + hkv * (d // 32) * 2
        elif is8:
            per_pos += hkv * d + hkv * (d // gs) * 2
        else:
            per_pos += hkv * d * 2
    n = ctx * per_pos + h * d * 2 + h * d * 4
    if append:
        n += 2 * hkv * d * 2 + per_pos
    return n


def decode_bytes(**kw):
    return step_bytes(append=False, **kw)


# --------------------------------------------------------------------------- helpers
def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 9 and f[1].replace(".", "").isdigit():
                    rows.append(f)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(float(r[2]) for r in rows),
                "reasons": reasons, "samples": len(rows)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(x, world):
    """Max of a host float over all ranks (NCCL on the GPUs, gloo on the CPU)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------- device state
class DecodeState:
    """R copies of the workload's pool (one physical page range per copy)."""

    def __init__(self, w, ctx, variant, copies, append_token=True):
        import torch

        from int8_kv_cache_02_gb300 import binding, inputs
        self.torch, self.binding = torch, binding
        self.ctx, self.copies = ctx, copies
        n_pages_copy = -(-ctx // PS)
        hkv, d, gs = w["Hkv"], w["D"], w["gs"]
        self.h = w["H"]
        self.pool = binding.KVPool(1, hkv, d, gs, PS, n_pages_copy * copies, variant)
        pts = []
        for c in range(copies):                              # disjoint page range per copy
            pt, _ = inputs.page_table([ctx], PS, seed=100 + c)
            pts.append(pt + c * n_pages_copy)
        self.pt = torch.cat(pts).cuda()                      # [copies][pages]
        n_cached = ctx - 1 if append_token else ctx
        kd = w["k"][:n_cached].reshape(1, n_cached, hkv, d).cuda()
        vd = w["v"][:n_cached].reshape(1, n_cached, hkv, d).cuda()
        zero = torch.zeros(1, dtype=torch.int32, device="cuda")
        for c in range(copies):
            binding.kv_quant_append(self.pool, 0, kd, vd, zero, self.pt[c:c + 1])
        del kd, vd
        self.k_new = w["k"][ctx - 1:ctx].reshape(1, 1, hkv, d).cuda()
        self.v_new = w["v"][ctx - 1:ctx].reshape(1, 1, hkv, d).cuda()
        self.pos = torch.tensor([ctx - 1], dtype=torch.int32, device="cuda")
        self.lens = torch.tensor([ctx], dtype=torch.int32, device="cuda")
        self.q = w["q"].cuda()
        self.out = torch.zeros((1, self.h, d), dtype=torch.float32, device="cuda")
        self.n_splits = binding.attn_decode_n_splits(self.pool, 1, ctx)
        self.ws = self.pool.decode_workspace(1, self.h, self.n_splits)
        self.append_token = append_token
        torch.cuda.synchronize()

    def step(self, c, append=True, decode=True):
        """append only, decode only, or both (one fused kernel: attn_decode_append_int8)."""
        b = self.binding
        pt = self.pt[c:c + 1]
        if append and decode and self.append_token:
            b.attn_decode_append_int8(self.pool, 0, self.q, self.k_new[0], self.v_new[0],
                                      self.lens, pt, self.out, self.ws, n_splits=self.n_splits)
            return
        if append and self.append_token:
            b.kv_quant_append(self.pool, 0, self.k_new, self.v_new, self.pos, pt)
        if decode:
            b.attn_decode_int8(self.pool, 0, self.q, self.lens, pt, self.out, self.ws,
                               n_splits=self.n_splits)

    def graph(self, n_steps, start=0, append=True, decode=True):
        torch = self.torch
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for i in range(3):                               # eager warm-up on the capture stream
                self.step((start + i) % self.copies, append, decode)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n_steps):
                self.step((start + i) % self.copies, append, decode)
        torch.cuda.synchronize()
        return g


def time_graph(g, reps=5):
    """Median over `reps` timed replays of graph `g` (ms per replay), after one
    untimed replay.  Before each timed replay the stream first runs a short
    device-side sleep, so that the graph is already submitted when the start
    event fires: the events then bracket the graph's kernels only, not the
    host's submission of the graph."""
    import torch
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        torch.cuda._sleep(100_000)          # ~50 us at 2 GHz: covers the graph submission
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times)


def l2_bytes():
    import torch
    try:
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except Exception:
        return 129 * 2 ** 20


def copies_for(bytes_per_copy):
    return max(2, math.ceil(2 * l2_bytes() / bytes_per_copy) + 1)


def traffic_from_profiles(kernel_src_sha):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_grouped8k.md")
    try:
        txt = open(path).read()
    except OSError:
        return None
    sha = val = None
    for line in txt.splitlines():
        if line.startswith("kernel source sha256:"):
            sha = line.split(":", 1)[1].strip()
        if line.startswith("dram bytes per launch:"):
            val = float(line.split(":", 1)[1].strip())
    return val if sha == kernel_src_sha and val is not None else None


DECODE_SOURCES = ("common.cuh", "decode_combine.cu", "decode_common.cuh", "decode_mma.cu",
                  "internal.h", "mma_common.cuh", "ptx.cuh", "q4_row.cuh", "quant_row.cuh")


def strip_comments(src):
    """C/C++ source without its comments and blank lines (string and character
    literals kept), so that a comment-only edit keeps a profile's source stamp."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).splitlines()]
    return "\n".join(ln for ln in lines if ln.strip())


def source_sha(names):
    """Hash of the comment-stripped sources `names` (files of csrc/)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "int8_kv_cache_02_gb300", "csrc")
    for n in names:
        h.update(strip_comments(open(os.path.join(csrc, n)).read()).encode())
    return h.hexdigest()[:16]


def decode_source_sha():
    """Source stamp of the timed decode step's kernels (the warp-level
    tensor-core decode kernel and the combine)."""
    return source_sha(DECODE_SOURCES)


# --------------------------------------------------------------------------- oracle timing
ORACLE_SNIPPET = r"""
import json, sys, time
sys.path.insert(0, {root!r})
from int8_kv_cache_02_gb300 import inputs
from oracle import pool as opool, attention as oatt
budget, max_steps, n_pos = {budget}, {max_steps}, {n_pos}
w = inputs.grouped8k()
pt, n = inputs.page_table([8192], 64)
P = opool.Pool(1, 2, 256, 64, 64, n, 0)
P.append_contiguous(0, w["k"][:8191].numpy(), w["v"][:8191].numpy(), 0, pt[0].numpy())
kn, vn, q = w["k"][8191:].numpy()[None], w["v"][8191:].numpy()[None], w["q"][0].numpy()
ptn = pt.numpy()
def step():
    P.append(0, kn, vn, [8191], ptn)
    kh, vh = P.gather_range(0, ptn[0], 8192 - n_pos, 8192)
    return oatt.decode(q, kh, vh, n_pos)
for _ in range({warmup}):
    step()
t0 = time.perf_counter(); k = 0
while k < max_steps and (k == 0 or time.perf_counter() - t0 < budget):
    step(); k += 1
print(json.dumps({{"steps": k, "seconds": time.perf_counter() - t0}}))
"""


def run_oracle(budget_s, max_steps, n_pos, warmup):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = ORACLE_SNIPPET.format(root=ROOT, budget=budget_s, max_steps=max_steps, n_pos=n_pos,
                                 warmup=warmup)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("oracle run failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def host_info():
    """The host the oracle runs on: its CPU model (from /proc/cpuinfo, else the
    platform's name for it) and the cores this process may run on."""
    import platform
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:   # Arm hosts name the core in lscpu, not in /proc/cpuinfo
        import subprocess
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name:"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    try:
        avail = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        avail = os.cpu_count()
    return {"cpu": model or platform.processor() or platform.machine(), "machine": platform.machine(),
            "cores_available": avail, "cores_used_by_the_oracle": 1}


def oracle_sample_bytes(n_pos):
    """Bytes of the sampled step: append + decode of all heads over the last n_pos positions."""
    return step_bytes(ctx=n_pos)


# --------------------------------------------------------------------------- arms
def run_ours(args, rank, world, local):
    import torch

    from int8_kv_cache_02_gb300 import binding, build, inputs
    build.build()
    torch.cuda.set_device(local)
    binding.lib()
    w = inputs.grouped8k()
    per_copy = decode_bytes()
    copies = args.copies or copies_for(per_copy)
    st = DecodeState(w, CTX, binding.K8V8, copies)
    K, W = args.steps, args.warmup

    g_warm = st.graph(W)
    g_step = st.graph(K, start=W)
    g_dec = st.graph(K, start=W, append=False)             # decode kernel alone
    g_warm.replay()
    torch.cuda.synchronize()

    barrier(world)
    with ClockSampler(local) as clk:
        ms = time_graph(g_step)
        ms_dec = time_graph(g_dec)
    ms = max_over_ranks(ms, world)
    ms_dec = max_over_ranks(ms_dec, world)
    barrier(world)
    clocks = clk.summary()

    ms_step = ms / K
    value = step_bytes() * K * world / (ms * 1e-3) / 1e9
    dec_s = ms_dec / K * 1e-3
    peak, peak_kind = measured_peaks()
    achieved = decode_bytes() / dec_s / 1e9
    src_sha = decode_source_sha()
    traffic = traffic_from_profiles(src_sha)

    # end to end through the public API: the step's inputs (q, new K row, new V
    # row) packed in one pinned host buffer and copied in, the output copied out
    nq, nk = st.q.numel(), st.k_new.numel()
    hin = torch.cat([w["q"].reshape(-1), st.k_new.cpu().reshape(-1),
                     st.v_new.cpu().reshape(-1)]).pin_memory()
    hout = torch.empty((1, H, D), dtype=torch.float32).pin_memory()
    din = torch.empty_like(hin, device="cuda")
    dq = din[:nq].view(st.q.shape)
    dk = din[nq:nq + nk].view(st.k_new.shape)
    dv = din[nq + nk:].view(st.v_new.shape)
    n_e2e = max(50, min(K, 500))

    def e2e_issue(c):
        din.copy_(hin, non_blocking=True)
        pt = st.pt[c:c + 1]
        binding.attn_decode_append_int8(st.pool, 0, dq, dk[0], dv[0], st.lens, pt, st.out, st.ws,
                                        n_splits=st.n_splits)
        hout.copy_(st.out, non_blocking=True)

    def e2e_time(run):
        for i in range(5):
            run(i % copies)
        barrier(world)
        t0 = time.perf_counter()
        for i in range(n_e2e):
            run(i % copies)
        return max_over_ranks(time.perf_counter() - t0, world)

    def eager_step(c):
        e2e_issue(c)
        torch.cuda.current_stream().synchronize()

    # as a serving loop runs it: one captured graph per pool copy holds the H2D copy
    # of the packed inputs, the public call and the D2H copy of the output; every
    # step replays one and waits for it
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        e2e_issue(0)
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    e2e_graphs = []
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            e2e_issue(c)
        e2e_graphs.append(g)
    torch.cuda.synchronize()

    def graph_step(c):
        e2e_graphs[c].replay()
        torch.cuda.current_stream().synchronize()

    e2e_s = e2e_time(graph_step)
    e2e_eager_s = e2e_time(eager_step)
    h2d = hin.numel() * 2
    d2h = hout.numel() * 4

    # correctness of what was timed: the last output against the first eager run
    ref = st.out.clone()
    st.step(0)
    torch.cuda.synchronize()
    assert torch.equal(ref, st.out), "decode output changed between runs"
    assert binding.kv_pool_read_device_error(st.pool) == 0

    extra = {}
    if not args.no_extra:
        extra = run_extra(args)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        r = run_oracle(budget_s=10.0, max_steps=1000, n_pos=CTX, warmup=1)
        cpu = {"value": step_bytes() * r["steps"] / r["seconds"] / 1e9, "unit": "GB/s",
               "cores": 1, "kind": "oracle",
               "sample": f"{r['steps']} full decode steps of the same workload (append + fp64 "
                         f"decode over 8192 positions, all 16 heads), single thread, "
                         f"{r['seconds']:.1f} s",
               "host": host_info()}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": ms_step, "us_per_step": ms_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "s8 codes + f16 scales in, f32 compute", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": B, "n_heads": H, "n_kv_heads": HKV,
                   "head_dim": D, "group_size": GS, "ctx": CTX, "page_size": PS,
                   "n_splits": st.n_splits, "pool_copies": copies,
                   "l2": f"inputs larger than L2: {copies} rotating pool copies "
                         f"({copies * per_copy / 2**20:.0f} MiB, L2 {l2_bytes() / 2**20:.0f} MiB)",
                   "timing": "CUDA graph of K steps, CUDA events on the launching stream",
                   "parallelism": f"replicas x{world}"},
        "attn_tokens_per_s": B * 1e3 / ms_step * world,
        "kv_positions_per_s": B * CTX * 1e3 / ms_step * world,
        "pct_of_8tbs": round(100 * value / world / 8000, 1),
        "e2e": {"value": round(step_bytes() * n_e2e * world / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": e2e_s / n_e2e * 1e6, "steps": n_e2e,
                "how": "host-timed; each step replays a captured graph of the H2D copy of the "
                       "packed inputs (pinned), attn_decode_append_int8 and the D2H copy of the "
                       "output, then synchronizes",
                "eager": {"value": round(step_bytes() * n_e2e * world / e2e_eager_s / 1e9, 2),
                          "us_per_step": e2e_eager_s / n_e2e * 1e6,
                          "how": "the same three calls issued from Python every step"}},
        "roofline": {"bound": "hbm", "kernel": "the attn_decode_int8 call: decode_mma_kernel "
                                               "(split-K partials) + decode_combine_kernel",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "traffic": traffic, "algorithmic_bytes": decode_bytes(),
                     "us_per_launch": dec_s * 1e6, "kernel_src_sha": src_sha},
        # per step: the fused append + decode kernel, and the combine kernel when
        # there are more than 8 splits (up to 8 combine inside the decode kernel)
        "gpu_launches": K * (2 if st.n_splits > 8 else 1),
        "clocks": clocks,
        "cpu_baseline": cpu,
        "extra": extra,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


PREFILL_FLOPS = 2 * 2 * 16 * 256 * sum(32768 + i + 1 for i in range(256))   # causal QK^T + PV


def run_prefill(n_iter=20):
    """Prefill chunk: append 256 new tokens (quantize) and causal attention of their
    queries over 33,024 positions; 16 query heads, 2 kv heads, head_dim 256."""
    import torch

    from int8_kv_cache_02_gb300 import binding, inputs
    w = inputs.prefill()
    start, n_new = w["start"], w["n_new"]
    L = start + n_new
    pt, n_pages = inputs.page_table([L], PS, seed=6)
    pool = binding.KVPool(1, 2, 256, 64, PS, n_pages, binding.K8V8)
    ptd = pt.cuda()
    kd = w["k"].reshape(1, L, 2, 256).cuda()
    vd = w["v"].reshape(1, L, 2, 256).cuda()
    binding.kv_quant_append(pool, 0, kd[:, :start].contiguous(), vd[:, :start].contiguous(),
                            torch.zeros(1, dtype=torch.int32, device="cuda"), ptd)
    kc, vc = kd[:, start:].contiguous(), vd[:, start:].contiguous()
    pos = torch.tensor([start], dtype=torch.int32, device="cuda")
    q = w["q"].cuda()
    ns = binding.attn_prefill_n_splits(pool, n_new, 16, start)
    ws = torch.empty(max(16, binding.attn_prefill_workspace_bytes(n_new, 16, 2, 256, ns)),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((n_new, 16, 256), dtype=torch.float32, device="cuda")

    def step():
        binding.kv_quant_append(pool, 0, kc, vc, pos, ptd)
        binding.attn_prefill_chunk_int8(pool, 0, q, start, ptd[0], out, ws, n_splits=ns)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(n_iter):
            step()
    ms = time_graph(g) / n_iter
    kv_bytes = L * 2 * (256 + 4 * 2) * 2
    tf = PREFILL_FLOPS / (ms * 1e-3) / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tpeak, tkind = float(json.load(f)["bf16_tflops"]), "measured bf16 burst (fp16: same nominal rate)"
    except Exception:
        tpeak, tkind = 1900.0, "fallback"
    return {"us_per_step": ms * 1e3, "TFLOPs": tf, "frac_of_tensor_peak": round(tf / tpeak, 4),
            "peak_source": tkind,
            "algorithmic_flops": PREFILL_FLOPS, "kv_bytes": kv_bytes, "n_splits": ns,
            "note": "append of the 256-token chunk + causal attention; the 33,024-position "
                    "cache (34 MB) is L2-resident; paced by the CUDA-core work between the two MMA batches of a page"}


def graph_us(issue, n_iter):
    """Median µs per call of `issue(i)` (i = 0 .. n_iter-1) replayed from a CUDA graph."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(3):
            issue(i)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n_iter):
            issue(i)
    return time_graph(g) / n_iter * 1e3


def rate(byt, us, l2):
    peak, kind = measured_peaks()
    gbs = byt / (us * 1e-6) / 1e9
    return {"us_per_step": us, "GBps": gbs, "frac_of_peak": round(gbs / peak, 4),
            "peak_source": kind, "algorithmic_bytes": byt, "l2": l2}


def run_batched(n_iter=20, window_copies=4):
    """Batched decode over a paged pool: 64 sequences, lengths uniform in [1024, 32768]
    (seed 3), 32 query / 8 kv heads, head_dim 128, one scale per (position, kv head);
    layer 0 full context, and the 512-position window layer held in `window_copies`
    copies (layers 1..) so that each replay reads HBM.  K/V are N(0,1) fp16 drawn
    on the device from seeded generators (the parity tests draw the same shapes on
    the CPU; the timing depends only on the shapes)."""
    import torch

    from int8_kv_cache_02_gb300 import binding, inputs
    lens, qs = inputs.batched_lengths_and_q()
    lens = [int(x) for x in lens]
    pt, n_pages = inputs.page_table(lens, PS, seed=11)
    n_layers = 1 + window_copies
    pool = binding.KVPool(n_layers, 8, 128, 128, PS, n_pages, binding.K8V8)
    ptd = pt.cuda()
    g = torch.Generator(device="cuda")
    for layer in range(n_layers):
        for b, L in enumerate(lens):
            g.manual_seed(5_000_000 + 1000 * layer + b)
            start = 0 if layer == 0 else max(0, L - 512)
            n = L - start
            k = torch.randn((1, n, 8, 128), generator=g, device="cuda").half()
            v = torch.randn((1, n, 8, 128), generator=g, device="cuda").half()
            binding.kv_quant_append(pool, layer, k, v,
                                    torch.tensor([start], dtype=torch.int32, device="cuda"),
                                    ptd[b:b + 1])
    torch.cuda.synchronize()
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = torch.empty((64, 32, 128), dtype=torch.float32, device="cuda")
    res = {"total_ctx": sum(lens), "inputs": "device-drawn N(0,1) fp16, seeded"}
    per_pos = 8 * 128 * 2 + 8 * 2 * 2        # int8 K, V rows + fp16 scales, all kv heads
    qo = 64 * 32 * 128 * (2 + 4)
    for name, window, layers in (("layer0_full", 0, [0]),
                                 ("layer1_window512", 512, list(range(1, n_layers)))):
        ns = binding.attn_decode_n_splits(pool, 64, window + PS if window else pt.shape[1] * PS)
        ws = pool.decode_workspace(64, 32, ns)
        q = qs[0 if window == 0 else 1].cuda()

        def issue(i, window=window, layers=layers, ns=ns, ws=ws, q=q):
            binding.attn_decode_int8(pool, layers[i % len(layers)], q, lens_d, ptd, out, ws,
                                     window=window, n_splits=ns)

        us = graph_us(issue, n_iter)
        vis = sum(min(L, window) if window else L for L in lens)
        l2 = ("pool 4.5 GB per layer: HBM-resident" if not window else
              f"{len(layers)} copies of the window layer ({len(layers) * vis * per_pos / 2**20:.0f} "
              f"MiB) rotated: HBM-resident")
        res[name] = dict(rate(vis * per_pos + qo, us, l2), n_splits=ns)
    del pool
    torch.cuda.empty_cache()
    return res


def run_tiny():
    """Tiny decode (batch 1, 8/2 heads, head_dim 128, 512 positions, one scale per
    (position, kv head)) at 4 splits and a single pass.  272 KB: L2-resident and
    bound by launch latency, not by HBM."""
    import torch

    from int8_kv_cache_02_gb300 import binding, inputs
    w = inputs.tiny()
    pt, n_pages = inputs.page_table([512], PS, seed=0)
    pool = binding.KVPool(1, 2, 128, 128, PS, n_pages, binding.K8V8)
    binding.kv_quant_append(pool, 0, w["k"].reshape(1, 512, 2, 128).cuda(),
                            w["v"].reshape(1, 512, 2, 128).cuda(),
                            torch.zeros(1, dtype=torch.int32, device="cuda"), pt.cuda())
    q, ptd = w["q"].cuda(), pt.cuda()
    lens = torch.tensor([512], dtype=torch.int32, device="cuda")
    out = torch.empty((1, 8, 128), dtype=torch.float32, device="cuda")
    byt = decode_bytes(ctx=512, hkv=2, h=8, d=128, gs=128)
    res = {}
    for ns in (4, 1):
        ws = pool.decode_workspace(1, 8, ns)
        us = graph_us(lambda i, ws=ws, ns=ns: binding.attn_decode_int8(
            pool, 0, q, lens, ptd, out, ws, n_splits=ns), 200)
        res[f"n_splits{ns}"] = rate(byt, us, "272 KB: L2-resident, launch-bound")
    return res


def run_windows(st, ctx, q_lens=(2, 4), n_iter=40):
    """Query windows (speculative verify) over a DecodeState's rotating pools:
    q_len queries per sequence, causal within the window."""
    import torch

    from int8_kv_cache_02_gb300 import binding
    res = {}
    for ql in q_lens:
        gq = torch.Generator(device="cuda").manual_seed(77 + ql)
        qw = torch.randn((1, ql, st.h, D), generator=gq, device="cuda").half()
        outw = torch.empty((1, ql, st.h, D), dtype=torch.float32, device="cuda")
        ns = binding.attn_decode_n_splits(st.pool, -(-ql * (st.h // HKV) // 8), ctx)
        ws = st.pool.decode_workspace(ql, st.h, ns)

        def issue(i, qw=qw, outw=outw, ns=ns, ws=ws):
            c = i % st.copies
            binding.attn_decode_multi_int8(st.pool, 0, qw, st.lens, st.pt[c:c + 1], outw, ws,
                                           n_splits=ns)

        us = graph_us(issue, n_iter)
        byt = decode_bytes(ctx=ctx) + (ql - 1) * H * D * 6
        res[f"q_len{ql}"] = dict(rate(byt, us, f"{st.copies} rotating pool copies"), n_splits=ns,
                                 attn_tokens_per_s=ql * 1e6 / us)
    return res


def run_extra(args):
    """Every workload besides the headline step: the tiny decode, the 128K-context
    decode (k8v8 and k8v16), query windows at 8K and 128K, the 64-sequence batch
    (both layers) and the prefill chunk.  Decode calls alone, L2 defeated by
    rotating copies where the data would fit in it."""
    import torch

    from int8_kv_cache_02_gb300 import binding, inputs
    out = {"tiny_512": run_tiny()}
    w = inputs.grouped8k()
    st = DecodeState(w, CTX, binding.K8V8, copies_for(decode_bytes()), append_token=False)
    out["grouped8k_windows"] = run_windows(st, CTX)
    del st
    torch.cuda.empty_cache()
    w = inputs.long128k()
    for name, variant, vi8 in (("long128k_k8v8", binding.K8V8, True),
                               ("long128k_k8v16", binding.K8V16, False)):
        per = decode_bytes(ctx=131072, v_int8=vi8)
        copies = max(2, math.ceil(2 * l2_bytes() / per) + 1)
        st = DecodeState(w, 131072, variant, copies, append_token=False)
        n = 60
        g = st.graph(n, append=False)
        us = time_graph(g) / n * 1e3
        out[name] = dict(rate(per, us, f"{copies} rotating pool copies"), n_splits=st.n_splits,
                         copies=copies)
        if vi8:
            out["long128k_windows"] = run_windows(st, 131072, n_iter=20)
        del st, g
        torch.cuda.empty_cache()
    # k8v4 (V rotated + Q4_0; tensor-core decode kernel) at 8K and 128K
    for name, wf, ctx in (("grouped8k_k8v4", inputs.grouped8k, CTX),
                          ("long128k_k8v4", inputs.long128k, 131072)):
        per = decode_bytes(ctx=ctx, v_int8=False, v_q4=True)
        copies = max(2, math.ceil(2 * l2_bytes() / per) + 1)
        st = DecodeState(wf(), ctx, binding.K8V4, copies, append_token=False)
        n = 40
        g = st.graph(n, append=False)
        us = time_graph(g) / n * 1e3
        out[name] = dict(rate(per, us, f"{copies} rotating pool copies"), n_splits=st.n_splits,
                         kernel="decode_mma_kernel (4-bit V) + decode_combine_kernel")
        del st, g
        torch.cuda.empty_cache()
    # q4_0 (K and V rotated + Q4_0; CUDA-core decode kernel) at 8K and 128K
    for name, wf, ctx in (("grouped8k_q4_0", inputs.grouped8k, CTX),
                          ("long128k_q4_0", inputs.long128k, 131072)):
        per = decode_bytes(ctx=ctx, k_int8=False, v_int8=False, k_q4=True, v_q4=True)
        copies = max(2, math.ceil(2 * l2_bytes() / per) + 1)
        st = DecodeState(wf(), ctx, binding.Q4_0, copies, append_token=False)
        n = 20
        g = st.graph(n, append=False)
        us = time_graph(g) / n * 1e3
        out[name] = dict(rate(per, us, f"{copies} rotating pool copies"), n_splits=st.n_splits,
                         kernel="decode_simt_kernel (4-bit K and V) + decode_combine_kernel")
        del st, g
        torch.cuda.empty_cache()
    if not getattr(args, "no_batched", False):
        out["batched_64seq"] = run_batched()
    out["prefill_chunk"] = run_prefill()
    return out


PROFILE_CASES = ("decode8k", "decode128k", "append256", "batched16", "prefill", "k8v4_8k",
                 "q4_0_8k", "simt_k8v4_8k", "tiny512", "window8k")


def run_profile_case(name, reps=5):
    """Set up one workload and issue its call `reps` times, eagerly, with no
    timing: the commands the ncu summaries under profiles/ are taken with.
      decode8k    attn_decode_append_int8 on the 8K workload (decode + combine)
      decode128k  attn_decode_int8 on the 128K workload, k8v8 (decode + combine)
      append256   kv_quant_append of the prefill chunk's 256 tokens
      batched16   attn_decode_int8 over 16 of the 64-sequence batch's sequences
                  (head_dim 128, the same lengths; 1.1 GB instead of 4.5 GB)
      prefill     append + attn_prefill_chunk_int8 of the 256-query chunk
      k8v4_8k     attn_decode_int8 on the 8K workload in a k8v4 pool
      q4_0_8k     the same in a q4_0 pool
      simt_k8v4_8k  the k8v4 case on the CUDA-core decode kernel
      tiny512     attn_decode_int8 on the 512-position workload (head_dim 128), 4 splits
      window8k    attn_decode_multi_int8 on the 8K workload, windows of 4 queries"""
    import torch

    from int8_kv_cache_02_gb300 import binding, inputs
    if name in ("decode8k", "k8v4_8k", "q4_0_8k", "simt_k8v4_8k"):
        w = inputs.grouped8k()
        variant = {"decode8k": binding.K8V8, "q4_0_8k": binding.Q4_0}.get(name, binding.K8V4)
        st = DecodeState(w, CTX, variant, 3, append_token=name == "decode8k")
        if name == "simt_k8v4_8k":
            st.pool.set_decode_kernel(binding.DECODE_SIMT)
        for i in range(reps):
            st.step(i % 3, append=name == "decode8k")
    elif name == "decode128k":
        st = DecodeState(inputs.long128k(), 131072, binding.K8V8, 3, append_token=False)
        for i in range(reps):
            st.step(i % 3, append=False)
    elif name == "append256":
        w = inputs.prefill()
        start, n_new = w["start"], w["n_new"]
        pt, n_pages = inputs.page_table([start + n_new], PS, seed=6)
        pool = binding.KVPool(1, 2, 256, 64, PS, n_pages, binding.K8V8)
        kc = w["k"][start:].reshape(1, n_new, 2, 256).cuda()
        vc = w["v"][start:].reshape(1, n_new, 2, 256).cuda()
        pos = torch.tensor([start], dtype=torch.int32, device="cuda")
        for _ in range(reps):
            binding.kv_quant_append(pool, 0, kc, vc, pos, pt.cuda())
    elif name == "batched16":
        lens, qs = inputs.batched_lengths_and_q()
        lens = [int(x) for x in lens[:16]]
        pt, n_pages = inputs.page_table(lens, PS, seed=11)
        pool = binding.KVPool(1, 8, 128, 128, PS, n_pages, binding.K8V8)
        ptd = pt.cuda()
        g = torch.Generator(device="cuda")
        for b, L in enumerate(lens):
            g.manual_seed(5_000_000 + b)
            k = torch.randn((1, L, 8, 128), generator=g, device="cuda").half()
            v = torch.randn((1, L, 8, 128), generator=g, device="cuda").half()
            binding.kv_quant_append(pool, 0, k, v, torch.zeros(1, dtype=torch.int32, device="cuda"),
                                    ptd[b:b + 1])
        lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
        ns = binding.attn_decode_n_splits(pool, 16, pt.shape[1] * PS)
        ws = pool.decode_workspace(16, 32, ns)
        out = torch.empty((16, 32, 128), dtype=torch.float32, device="cuda")
        q = qs[0][:16].contiguous().cuda()
        for _ in range(reps):
            binding.attn_decode_int8(pool, 0, q, lens_d, ptd, out, ws, n_splits=ns)
    elif name == "prefill":
        run_prefill(n_iter=reps)
    elif name == "tiny512":
        w = inputs.tiny()
        pt, n_pages = inputs.page_table([512], PS, seed=0)
        pool = binding.KVPool(1, 2, 128, 128, PS, n_pages, binding.K8V8)
        binding.kv_quant_append(pool, 0, w["k"].reshape(1, 512, 2, 128).cuda(),
                                w["v"].reshape(1, 512, 2, 128).cuda(),
                                torch.zeros(1, dtype=torch.int32, device="cuda"), pt.cuda())
        out = torch.empty((1, 8, 128), dtype=torch.float32, device="cuda")
        ws = pool.decode_workspace(1, 8, 4)
        lens = torch.tensor([512], dtype=torch.int32, device="cuda")
        for _ in range(reps):
            binding.attn_decode_int8(pool, 0, w["q"].cuda(), lens, pt.cuda(), out, ws, n_splits=4)
    elif name == "window8k":
        st = DecodeState(inputs.grouped8k(), CTX, binding.K8V8, 3, append_token=False)
        g = torch.Generator().manual_seed(70)
        qw = inputs.normal_f16((1, 4, st.h, D), g).cuda()
        outw = torch.empty((1, 4, st.h, D), dtype=torch.float32, device="cuda")
        ns = binding.attn_decode_n_splits(st.pool, 4, CTX)
        ws = st.pool.decode_workspace(4, st.h, ns)
        for i in range(reps):
            binding.attn_decode_multi_int8(st.pool, 0, qw, st.lens, st.pt[i % 3:i % 3 + 1], outw, ws,
                                           n_splits=ns)
    else:
        raise SystemExit(f"unknown profile case {name}; one of {', '.join(PROFILE_CASES)}")
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": name, "reps": reps}), flush=True)


def run_reference(args, rank, world, local):
    if rank != 0:
        return
    K, W = args.steps, args.warmup
    probe = run_oracle(budget_s=1e9, max_steps=2, n_pos=CTX, warmup=1)
    t_full = probe["seconds"] / max(1, probe["steps"])
    frac = min(1.0, 60.0 / max(1e-9, K * t_full))
    n_pos = max(PS, int(CTX * frac) // PS * PS)
    r = run_oracle(budget_s=1e9, max_steps=K, n_pos=n_pos, warmup=W)
    byt = oracle_sample_bytes(n_pos)
    value = byt * r["steps"] / r["seconds"] / 1e9
    ms = r["seconds"] / r["steps"] * 1e3
    sample = (f"each step: append 1 token + fp64 decode of all 16 heads over the last {n_pos} "
              f"of the 8192 positions (single thread)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": r["steps"], "warmup": W, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": B, "n_heads": H, "n_kv_heads": HKV,
                   "head_dim": D, "group_size": GS, "ctx": CTX, "sampled_positions": n_pos},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample, "host": host_info()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--copies", type=int, default=0, help="pool copies (0: enough to defeat L2)")
    ap.add_argument("--no-extra", action="store_true", help="skip the 128K measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle timing")
    ap.add_argument("--no-batched", action="store_true",
                    help="skip the 64-sequence paged batch among the extra workloads")
    ap.add_argument("--extra-only", action="store_true",
                    help="run only the extra workloads and print them (profiling aid)")
    ap.add_argument("--profile-case", choices=PROFILE_CASES,
                    help="set up one workload and issue its call a few times, untimed "
                         "(the commands of the ncu summaries under profiles/)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if args.impl == "ours":
            import torch
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    try:
        if args.profile_case:
            import torch

            from int8_kv_cache_02_gb300 import build
            build.build()
            torch.cuda.set_device(local)
            run_profile_case(args.profile_case)
        elif args.extra_only:
            import torch

            from int8_kv_cache_02_gb300 import build
            build.build()
            torch.cuda.set_device(local)
            res = run_extra(args)
            print(json.dumps(res), flush=True)
        elif args.impl == "reference":
            run_reference(args, rank, world, local)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
