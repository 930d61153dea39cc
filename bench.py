"""Benchmark of the NVFP4 paged-KV hot path on B300: plan -> quantize-append ->
causal prefill, through the C ABI of libfi_nvfp4.so.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload uniform|single|ragged|decode|decode_spec]
                    [--kv-format nvfp4|fp8]
                    [--no-e2e] [--no-cpu-baseline] [--no-extra]

One step is one pass of the whole path over one batch: fi_prefill_plan of the
batch (its upload enqueued first, so that the append and the prefill are
adjacent on the stream and the prefill is launched as the append's
programmatic dependent), fi_nvfp4_append of every token's K/V into the cache,
fi_prefill_run.  The default workload is the uniform batch: 1024 sequences of
qo_len = kv_len = 1024, H_q = 32, H_kv = 8, head_dim = 128, page_size = 16
(synthetic N(0,1) bf16 inputs, random page table).  `value` is the causal
prefill FLOPs of a step divided by the measured step time (TFLOP/s), timed over
K steps with no event between the kernels; a second pass of K steps with
events around each kernel gives the per-kernel times of `roofline` and
`append_in_step`.  The same run also measures, each in its own timed passes,
the single 2048 x 2048 prefill, the ragged batch, the 128 x 4096 decode (1 and
8 query tokens per sequence) and the FP8 (E4M3) variant of the uniform batch
(`workloads`), and the 8192-token
append with cold L2 (`append_bench`: 24 rotating buffer sets captured in one
CUDA graph).

Under torchrun (N > 1) every rank runs its own independent copy of the
workload on its own GPU (the path has no exchange step): scaling is weak and
`value` is the FLOPs of all ranks over the slowest rank's time.

--impl reference times the CPU oracle (the slow, plain C++ definition of the
method) on a fixed sample of the same workload, on the host cores; the
`cpu_baseline` leg of our arm times the same sample.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "causal prefill TFLOP/s over NVFP4 paged KV; append GB/s; % of roofline"
UNIT = "TFLOP/s"

WORKLOAD_DESC = {
    "uniform": "uniform batch: 1024 x (qo_len=kv_len=1024), H_q=32, H_kv=8, head_dim=128, "
               "page_size=16, NVFP4 paged KV, append + plan + causal prefill",
    "single": "single sequence 2048x2048, H_q=32, H_kv=8, head_dim=128, page_size=16, "
              "append + plan + causal prefill",
    "ragged": "ragged batch: 256 sequences, qo_len=kv_len log-uniform in [128,16384], H_q=32, "
              "H_kv=8, head_dim=128, page_size=16, append + plan + causal prefill",
    "decode": "decode batch: 128 sequences x kv_len 4096, qo_len 1, H_q=32, H_kv=8, "
              "head_dim=128, page_size=16, decode plan + append of the newest token + decode",
    "decode_spec": "speculative decode batch: 128 sequences x kv_len 4096, qo_len 8 (32 rows "
                   "per KV head), H_q=32, H_kv=8, head_dim=128, page_size=16, decode plan + "
                   "append of the newest 8 tokens + decode",
}

# Oracle sample (both arms): sequences of the workload drawn with a fixed seed
# until about ORACLE_TOKENS cache tokens, and at most ORACLE_ROWS of their
# (token, query head) rows in a seeded random order.
ORACLE_TOKENS = 8192
ORACLE_ROWS = 1 << 18


# ----------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def recorded_traffic(key):
    """DRAM bytes per launch recorded from an ncu capture (profiles/traffic.json),
    or None when the kernel's sources changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(key)
    if not rec:
        return None
    h = hashlib.sha256()
    for src in rec["sources"]:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return rec["dram_bytes_per_launch"] if h.hexdigest()[:16] == rec["source_sha256_16"] else None


def newest_token_rows(qo_indptr, kv_indptr):
    """Rows (in the kv_indptr layout) of each sequence's newest qo_len tokens: the
    tokens a decode step appends, the rest of the context being in the cache."""
    qlens = np.diff(np.asarray(qo_indptr))
    ends = np.asarray(kv_indptr)[1:]
    if len(ends) == 0:
        return np.zeros(0, np.int64)
    return np.concatenate([np.arange(e - q, e) for e, q in zip(ends, qlens)]).astype(np.int64)


def append_bytes(num_tokens_written, num_tokens_skipped, num_kv_heads, head_dim, fp8=False):
    """Algorithmic bytes of one append: per written token read K and V bf16
    rows, write K and V NVFP4 rows (codes + scales; FP8: one byte per
    element) and read its 8-byte slot; per skipped token read its slot; plus
    the two 4-byte scales."""
    row = head_dim if fp8 else head_dim // 2 + head_dim // 16
    per_tok = num_kv_heads * (2 * head_dim * 2) + num_kv_heads * 2 * row + 8
    return num_tokens_written * per_tok + num_tokens_skipped * 8 + 8


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- our arm
class PathRunner:
    """Device-resident inputs and outputs of one workload, and one step of the
    path (append -> plan -> run) through the C ABI."""

    def __init__(self, fi, name, device, seqs=0, kv_format="nvfp4"):
        self.fi = fi
        self.fp8 = kv_format == "fp8"
        sp = W.spec(name)
        if seqs:
            sp.seq_lens = sp.seq_lens[:seqs]
        self.sp = sp
        d = W.make(sp, device=device)
        self.d = d
        self.device = device
        self.k, self.v, self.q = d["k"], d["v"], d["q"]
        self.slots = d["slot_mapping"].to(device)
        self.page_table = d["page_table"].to(device)
        self.qo_indptr = d["qo_indptr"].numpy()
        self.kv_indptr = d["kv_indptr"].numpy()
        if self.fp8:
            # FP8 decode scales map each tensor's amax to 448
            ks = (self.k.float().abs().max() / 448.0).reshape(1).to(torch.float32)
            vs = (self.v.float().abs().max() / 448.0).reshape(1).to(torch.float32)
            self.cache = fi.FP8Cache(d["num_pages"], sp.num_kv_heads, sp.page_size, sp.head_dim,
                                     device=device, k_scale=ks, v_scale=vs, fill=0)
        else:
            ks = torch.tensor([d["k_scale"]], dtype=torch.float32, device=device)
            vs = torch.tensor([d["v_scale"]], dtype=torch.float32, device=device)
            self.cache = fi.NVFP4Cache(d["num_pages"], sp.num_kv_heads, sp.page_size,
                                       sp.head_dim, device=device, k_scale=ks, v_scale=vs, fill=0)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:2], dtype=torch.float32, device=device)
        self.ctx = fi.fi_context_create()
        self.plan = fi.fi_plan_create(self.ctx)
        self.decode = sp.attn == "decode"
        if self.decode:
            # A decode step appends each sequence's newest qo_len tokens; the
            # rest of its context is written into the cache once, here.
            append = fi.fi_fp8_append if self.fp8 else fi.fi_nvfp4_append
            append(self.ctx, self.k, self.v, self.cache.k_scale, self.cache.v_scale, self.slots,
                   self.cache)
            torch.cuda.synchronize()
            idx_t = torch.from_numpy(newest_token_rows(self.qo_indptr, self.kv_indptr)).to(device)
            self.k = self.k.index_select(0, idx_t).contiguous()
            self.v = self.v.index_select(0, idx_t).contiguous()
            self.slots = self.slots.index_select(0, idx_t).contiguous()
        lens = np.diff(self.qo_indptr).tolist()
        kv_lens = np.diff(self.kv_indptr).tolist()
        self.flops = W.causal_flops(lens, kv_lens, sp.num_qo_heads, sp.head_dim)
        # decode: HBM bytes the attention must move (the NVFP4 K and V of every
        # sequence once, Q in, O and LSE out)
        self.decode_bytes = (sum(kv_lens) * sp.num_kv_heads * 2 *
                             (sp.head_dim // 2 + sp.head_dim // 16) +
                             sum(lens) * sp.num_qo_heads * (2 * sp.head_dim * 2 + 4))
        self.tokens = int(self.qo_indptr[-1])
        self.append_bytes = append_bytes(self.tokens, 0, sp.num_kv_heads, sp.head_dim,
                                         fp8=self.fp8)

    def step(self, stream, ev=None):
        """plan (host planning, upload enqueued) -> append -> run.  With `ev`
        (three events) the append and the run are bracketed by events:
        ev[0] append ev[1] run ev[2]."""
        fi, sp = self.fi, self.sp
        if self.decode:
            fi.fi_decode_plan(self.plan, self.qo_indptr, self.kv_indptr, self.page_table,
                              sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size,
                              sm_scale=self.d["sm_scale"], stream=stream)
        else:
            fi.fi_prefill_plan(self.plan, self.qo_indptr, self.kv_indptr, self.page_table,
                               sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size,
                               sm_scale=self.d["sm_scale"], stream=stream,
                               kv_format=1 if self.fp8 else 0)
        if ev is not None:
            ev[0].record(stream)
        self.launch_append(stream)
        if ev is not None:
            ev[1].record(stream)
        self.launch_attention(stream)
        if ev is not None:
            ev[2].record(stream)

    def launch_append(self, stream):
        """The step's append (one kernel launch)."""
        fi = self.fi
        append = fi.fi_fp8_append if self.fp8 else fi.fi_nvfp4_append
        append(self.ctx, self.k, self.v, self.cache.k_scale, self.cache.v_scale, self.slots,
               self.cache, stream=stream)

    def launch_attention(self, stream):
        """The step's attention with the current plan (the decode adds its
        merge kernel when a sequence is split into chunks)."""
        fi = self.fi
        if self.decode:
            run = fi.fi_decode_run
        else:
            run = fi.fi_prefill_run_fp8 if self.fp8 else fi.fi_prefill_run
        run(self.plan, self.q, self.cache, self.out, self.lse, stream=stream)

    def launches_per_step(self):
        """Kernels of this library one step launches: the append and the
        attention (a decode with split sequences adds its merge kernel)."""
        if self.decode:
            info = self.fi.fi_plan_get_info(self.plan)
            merges = info["num_units"] > info["batch"] * self.sp.num_kv_heads
            return 3 if merges else 2
        return 2

    def status(self):
        return self.fi.fi_device_status(self.ctx)

    def close(self):
        self.fi.fi_plan_destroy(self.plan)
        self.fi.fi_context_destroy(self.ctx)


def barrier(dist_on):
    if dist_on:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, dist_on, device):
    if not dist_on:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(flops_per_rank, step_ms_max, world):
    """Whole-job throughput in TFLOP/s: every rank runs its own copy of the
    workload (weak scaling), so the FLOPs of all ranks over the slowest
    rank's step time."""
    return world * flops_per_rank / (step_ms_max * 1e-3) / 1e12


def time_device_steps(runner, stream, steps, warmup, dist_on, device):
    """Returns (step ms over `steps` steps with no event between the kernels,
    per-step append ms, per-step attention ms from a second pass of `steps`
    steps with events around each kernel)."""
    for _ in range(warmup):
        runner.step(stream)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(dist_on)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        runner.step(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(dist_on)
    total_ms = start.elapsed_time(end)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        runner.step(stream, evs[i])
    torch.cuda.synchronize()
    append_ms = [e[0].elapsed_time(e[1]) for e in evs]
    attn_ms = [e[1].elapsed_time(e[2]) for e in evs]
    return total_ms, append_ms, attn_ms


def time_launches(fn, stream, reps):
    """Per-launch device ms of `fn` (which enqueues one launch on `stream`):
    `reps` launches captured into one CUDA graph, one replay to warm up, then
    one replay timed with CUDA events on `stream`.  Inside the graph the
    launches follow one another with no host gap, which event pairs around
    single launches do not guarantee once a kernel is shorter than its host
    launch path (the decode step's kernels)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                fn(stream)
    g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    del g
    return ms


def time_e2e(runner, stream, steps, warmup):
    """Same step through the public API with host inputs: pinned host K/V/Q,
    slot_mapping and page_table are copied to the device inside the timed
    region, and the attention output (and LSE) are read back to pinned host
    memory at the end of every step.  Two device buffer sets alternate between
    steps, as a serving loop double-buffers its transfers: step s's inputs are
    copied on one copy stream while step s-1's kernels run, and step s-1's
    results are read back on another while step s's kernels run.  Every step
    still moves all of its inputs and results; the time per step is the whole
    timed region (first copy in to last copy out) over the steps.  Returns
    (seconds per step, bytes in per step, bytes out per step, the last step's
    host O and LSE)."""
    names = ("k", "v", "q", "slots", "page_table")
    host_in = {n: getattr(runner, n).cpu().pin_memory() for n in names}
    ho = torch.empty(runner.out.shape, dtype=runner.out.dtype, pin_memory=True)
    hl = torch.empty(runner.lse.shape, dtype=runner.lse.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    own = {n: getattr(runner, n) for n in names + ("out", "lse")}
    sets = [own, {n: torch.empty_like(t) for n, t in own.items()}]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    # per buffer set: inputs copied / kernels done / results read back
    ev = [{k: torch.cuda.Event() for k in ("in", "run", "out")} for _ in sets]
    for e in ev:
        for x in e.values():
            x.record(stream)
    n_step = [0]

    def one():
        b = sets[n_step[0] % 2]
        e = ev[n_step[0] % 2]
        n_step[0] += 1
        s_in.wait_event(e["run"])            # the previous kernels of this set have read it
        with torch.cuda.stream(s_in):
            for n in names:
                b[n].copy_(host_in[n], non_blocking=True)
        e["in"].record(s_in)
        stream.wait_event(e["in"])
        stream.wait_event(e["out"])          # this set's previous results are read back
        for n, t in b.items():
            setattr(runner, n, t)
        runner.step(stream)
        e["run"].record(stream)
        s_out.wait_event(e["run"])
        with torch.cuda.stream(s_out):
            ho.copy_(b["out"], non_blocking=True)
            hl.copy_(b["lse"], non_blocking=True)
        e["out"].record(s_out)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    for n, t in own.items():
        setattr(runner, n, t)
    del sets
    return dt / steps, h2d, d2h, (ho, hl)


def time_append_cold(fi, device, n_sets=24, reps=20):
    """Append of the 8192-token workload: n_sets distinct input / slot / cache
    buffer sets (together far larger than L2) appended back to back from one
    CUDA graph, as a model's per-layer appends run.  Returns per-append ms
    (cold L2) and the same append repeated on one set (warm L2)."""
    sp = W.spec("append")
    d = W.make(sp, device=device)
    ctx = fi.fi_context_create()
    ks = torch.tensor([d["k_scale"]], dtype=torch.float32, device=device)
    vs = torch.tensor([d["v_scale"]], dtype=torch.float32, device=device)
    sets = []
    for _ in range(n_sets):
        c = fi.NVFP4Cache(sp.num_pages, sp.num_kv_heads, sp.page_size, sp.head_dim,
                          device=device, k_scale=ks, v_scale=vs, fill=0)
        sets.append((d["k"].clone(), d["v"].clone(), d["slot_mapping"].to(device).clone(), c))
    set_bytes = sum(t.numel() * t.element_size() for t in sets[0][:3]) + \
        sum(t.numel() for t in (sets[0][3].k_data, sets[0][3].v_data, sets[0][3].k_sf,
                                 sets[0][3].v_sf))
    s = torch.cuda.Stream(device=device)
    s.wait_stream(torch.cuda.current_stream(device))  # inputs are made on the current stream
    for k, v, sl, c in sets:
        fi.fi_nvfp4_append(ctx, k, v, ks, vs, sl, c, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for k, v, sl, c in sets:
                fi.fi_nvfp4_append(ctx, k, v, ks, vs, sl, c, stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    cold_ms = e0.elapsed_time(e1) / (reps * n_sets)
    # warm: one set, back to back
    k, v, sl, c = sets[0]
    gw = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(gw, stream=s):
            for _ in range(n_sets):
                fi.fi_nvfp4_append(ctx, k, v, ks, vs, sl, c, stream=s)
    gw.replay()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(reps):
            gw.replay()
        e1.record(s)
    torch.cuda.synchronize()
    warm_ms = e0.elapsed_time(e1) / (reps * n_sets)
    status = fi.fi_device_status(ctx)
    fi.fi_context_destroy(ctx)
    n_skip = int((d["slot_mapping"] < 0).sum())
    nbytes = append_bytes(sp.append_tokens - n_skip, n_skip, sp.num_kv_heads, sp.head_dim)
    return {"cold_ms": cold_ms, "warm_ms": warm_ms, "bytes": nbytes, "status": status,
            "sets": n_sets, "set_bytes": set_bytes, "launches": n_sets * reps}


# ----------------------------------------------------------------- oracle legs
def time_plan_host(fi, device, reps=20):
    """Host time of one fi_prefill_plan / fi_decode_plan call (the call a user
    makes: host planning, the list copied into pinned staging, its upload
    enqueued), median over `reps` calls with the stream idle before each (a
    plan waits only when a third plan would reuse a staging buffer whose upload
    the stream has not reached).  Batches of 64, 256 and 1024 sequences, H_q=32,
    H_kv=8, D=128, page_size=16: uniform (1024 tokens each) and ragged (the
    ragged workload's length distribution, log-uniform in [128, 16384])."""
    ctx = fi.fi_context_create()
    plan = fi.fi_plan_create(ctx)
    out = {}
    for B in (64, 256, 1024):
        pt = torch.zeros((B, 16384 // 16), dtype=torch.int32, device=device)
        for kind in ("uniform", "ragged"):
            lens = np.full(B, 1024, np.int32) if kind == "uniform" else \
                np.array(W.ragged_lengths(B, 128, 16384, 4000), np.int32)
            ind = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
            calls = (("prefill", lambda: fi.fi_prefill_plan(plan, ind, ind, pt, 32, 8, 128, 16)),
                     ("decode", lambda: fi.fi_decode_plan(plan, np.arange(B + 1, dtype=np.int32),
                                                          ind, pt, 32, 8, 128, 16)))
            for what, call in calls:
                ts = []
                for _ in range(reps + 2):
                    torch.cuda.synchronize()
                    t0 = time.perf_counter()
                    call()
                    ts.append(time.perf_counter() - t0)
                out[f"{what}_{kind}_b{B}"] = float(np.median(ts[2:]) * 1e6)
    torch.cuda.synchronize()
    fi.fi_plan_destroy(plan)
    fi.fi_context_destroy(ctx)
    return out


def oracle_sample(name, seed=0):
    """Times the CPU oracle on a fixed sample of workload `name`: sequences
    drawn with `seed` (same per-sequence shapes, freshly drawn seeded inputs)
    until about ORACLE_TOKENS cache tokens, appended by the oracle into a host
    cache (plan-free: the oracle needs none), then the attention of at most
    ORACLE_ROWS of their (token, query head) rows in a seeded random order, in
    chunks.  Returns a dict: flops of the sampled rows, append and attention
    seconds, rows, threads and a description."""
    import oracle as O
    full = W.spec(name)
    n_seqs = max(1, min(full.batch, math.ceil(ORACLE_TOKENS * full.batch / sum(full.seq_lens))))
    sp = W.sample_spec(name, n_seqs, seed)
    d = W.make(sp, device="cpu")
    qo = d["qo_indptr"].numpy().astype(np.int64)
    kv = d["kv_indptr"].numpy().astype(np.int64)
    rng = np.random.default_rng(seed)
    threads = O.max_threads()
    host = O.new_cache(d["num_pages"], sp.num_kv_heads, sp.page_size, sp.head_dim, 0)
    t0 = time.perf_counter()
    st = O.append(W.bits(d["k"]), W.bits(d["v"]), d["k_scale"], d["v_scale"],
                  d["slot_mapping"].numpy(), host)
    t_append = time.perf_counter() - t0
    assert st == 0
    all_rows = np.stack(np.meshgrid(np.arange(int(qo[-1])), np.arange(sp.num_qo_heads),
                                    indexing="ij"), -1).reshape(-1, 2).astype(np.int64)
    rng.shuffle(all_rows)
    rows_all = all_rows[:ORACLE_ROWS]
    seq_of = np.searchsorted(qo, rows_all[:, 0], side="right") - 1
    i = rows_all[:, 0] - qo[seq_of]
    visible = i + (kv[seq_of + 1] - kv[seq_of]) - (qo[seq_of + 1] - qo[seq_of]) + 1
    flops = int(4 * sp.head_dim * visible.sum())
    qb = W.bits(d["q"])
    pt = d["page_table"].numpy()
    t_attn, chunk = 0.0, 65536
    for c0 in range(0, len(rows_all), chunk):
        t0 = time.perf_counter()
        O.prefill(qb, qo.astype(np.int32), kv.astype(np.int32), pt, host, sp.num_qo_heads,
                  d["k_scale"], d["v_scale"], d["sm_scale"], rows=rows_all[c0:c0 + chunk],
                  threads=threads)
        t_attn += time.perf_counter() - t0
    lens_txt = f"{len(sp.seq_lens)} x {sp.seq_lens[0]}" if len(set(sp.seq_lens)) == 1 \
        else f"{sum(sp.seq_lens)} tokens in total"
    desc = (f"{len(sp.seq_lens)} sequences of the workload ({lens_txt}): oracle append of "
            f"their K/V ({t_append:.2f} s) + fp64 attention of {len(rows_all)} (token, query "
            f"head) rows ({t_attn:.2f} s); value = the rows' causal FLOPs / (append + "
            f"attention time)")
    return {"flops": flops, "t_append": t_append, "t_attn": t_attn, "rows": len(rows_all),
            "threads": threads, "desc": desc}


def run_reference(args):
    """--impl reference: the oracle, timed on the host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    for i in range(args.warmup):
        oracle_sample(args.workload, seed=100 + i)
    tot_f, tot_t, res = 0, 0.0, None
    for i in range(args.steps):
        res = oracle_sample(args.workload, seed=i)
        tot_f += res["flops"]
        tot_t += res["t_append"] + res["t_attn"]
    value = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC[args.workload], "sampled": True},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": res["threads"],
                             "kind": "oracle", "sample": res["desc"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- main
def kernel_names(runner):
    """Names of the step's kernels: (append, attention)."""
    if runner.fp8:
        app = "fp8_append_kernel"
    else:
        # the library's switch to the staged kernel
        app = "nvfp4_append_staged_kernel" if runner.tokens >= 65536 else "nvfp4_append_kernel"
    attn = "nvfp4_decode_t_kernel" if runner.decode else "nvfp4_prefill_kernel"
    return app, attn


def measure(fi, name, device, steps, warmup, dist_on, kv_format="nvfp4", seqs=0):
    """Builds workload `name`, checks one clean step, times it; returns the
    runner and its numbers."""
    runner = PathRunner(fi, name, device, seqs, kv_format=kv_format)
    stream = torch.cuda.Stream(device=device)
    stream.wait_stream(torch.cuda.current_stream(device))  # inputs are made on the current stream
    # correctness guard: the step must run clean before it is timed
    runner.step(stream)
    st = runner.status()
    if st != 0:
        raise RuntimeError(f"{name}: device status {st} after the first step")
    total_ms, append_ms, attn_ms = time_device_steps(runner, stream, steps, warmup, dist_on,
                                                     device)
    # also the step's own append and attention (same plan and inputs), each
    # repeated back to back from a CUDA graph for about 40 ms: the kernel time
    # without the host gaps that the event pairs of the second pass can hold
    # when a kernel is shorter than its host launch path
    a_est, r_est = statistics.mean(append_ms), statistics.mean(attn_ms)
    app_ms = time_launches(runner.launch_append, stream, max(5, min(400, int(40 / max(a_est, 1e-3)))))
    att_ms = time_launches(runner.launch_attention, stream,
                           max(3, min(400, int(40 / max(r_est, 1e-3)))))
    st = runner.status()
    if st != 0:
        raise RuntimeError(f"{name}: device status {st} after the timed steps")
    return runner, stream, {"step_ms": total_ms / steps, "append_ms": a_est, "attn_ms": r_est,
                            "append_ms_b2b": app_ms, "attn_ms_b2b": att_ms}


def attention_entry(runner, t, peaks, traffic_key=None):
    """Per-launch numbers of the attention kernel of a measured workload;
    `traffic_key` names its recorded DRAM traffic (full-size workloads only)."""
    app_name, attn_name = kernel_names(runner)
    ms = t["attn_ms"]
    e = {"kernel": attn_name, "ms_per_launch": ms, "ms_per_launch_back_to_back": t["attn_ms_b2b"],
         "step_ms": t["step_ms"],
         "tflops": runner.flops / (ms * 1e-3) / 1e12,
         "step_tflops": runner.flops / (t["step_ms"] * 1e-3) / 1e12,
         "flops_per_launch": runner.flops}
    if runner.decode:
        gbs = runner.decode_bytes / (ms * 1e-3) / 1e9
        e.update({"bound": "hbm", "gbs": gbs, "algorithmic_bytes": runner.decode_bytes,
                  "frac": gbs / peaks["hbm_gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                  "traffic": recorded_traffic(traffic_key) if traffic_key else None})
    else:
        e.update({"bound": "tensor", "frac": e["tflops"] / peaks["bf16_tflops"],
                  "frac_of_sustained": e["tflops"] / peaks["bf16_tflops_sustained"],
                  "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"})
    app_gbs = runner.append_bytes / (t["append_ms"] * 1e-3) / 1e9
    e["append"] = {"kernel": app_name, "ms_per_launch": t["append_ms"],
                   "ms_per_launch_back_to_back": t["append_ms_b2b"], "gbs": app_gbs,
                   "frac": app_gbs / peaks["hbm_gbs"], "algorithmic_bytes": runner.append_bytes}
    return e


EXTRA = [("single", "single", "nvfp4"), ("ragged", "ragged", "nvfp4"),
         ("decode", "decode", "nvfp4"), ("decode_spec", "decode_spec", "nvfp4"),
         ("fp8_uniform", "uniform", "fp8")]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_DESC), default="uniform")
    ap.add_argument("--kv-format", choices=["nvfp4", "fp8"], default="nvfp4",
                    help="fp8: the FP8 (E4M3) paged KV variant of the same path")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-append-bench", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads (single, ragged, decode, decode_spec, fp8)")
    ap.add_argument("--extra-steps", type=int, default=10)
    ap.add_argument("--seqs", type=int, default=0,
                    help="use only the first N sequences of the workload (profiling cases)")
    ap.add_argument("--only", choices=["all", "append"], default="all",
                    help="append: run only the cold-L2 append measurement")
    args = ap.parse_args()
    if args.steps < 1 or args.warmup < 0:
        raise SystemExit("--steps >= 1 and --warmup >= 0")
    if args.impl == "reference":
        return run_reference(args)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist_on = world > 1
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if dist_on:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    import nvfp4_paged_kv_slot_b300 as fi
    peaks = load_peaks()
    if args.only == "append":
        a = time_append_cold(fi, device)
        gbs = a["bytes"] / (a["cold_ms"] * 1e-3) / 1e9
        print(json.dumps({"append_only": True, "gbs_cold_l2": gbs, "us_cold_l2": a["cold_ms"] * 1e3,
                          "us_warm_l2": a["warm_ms"] * 1e3, "frac": gbs / peaks["hbm_gbs"],
                          "status": a["status"]}), flush=True)
        return 0 if a["status"] == 0 else 1

    clocks = ClockSampler(local_rank)
    clocks.start()
    runner, stream, t = measure(fi, args.workload, device, args.steps, args.warmup, dist_on,
                                kv_format=args.kv_format, seqs=args.seqs)
    clk = clocks.stop()
    step_ms = max_over_ranks(t["step_ms"], dist_on, device)
    value = aggregate_value(runner.flops, step_ms, world)
    head = attention_entry(runner, t, peaks,
                           "decode_128x4096" if args.workload == "decode" and not args.seqs
                           else None)
    full_uniform = args.workload == "uniform" and not args.seqs and not runner.fp8
    traffic = recorded_traffic("prefill_uniform") if full_uniform else None
    if runner.decode:
        roofline = {"bound": "hbm", "achieved": head["gbs"], "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": head["frac"], "traffic": head["traffic"],
                    "kernel": head["kernel"], "algorithmic_bytes": runner.decode_bytes,
                    "ms_per_launch": head["ms_per_launch"],
                    "ms_per_launch_back_to_back": head["ms_per_launch_back_to_back"],
                    "peak_kind": f"HBM copy ({peaks['source']})"}
    else:
        roofline = {"bound": "tensor", "achieved": head["tflops"], "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": head["frac"], "traffic": traffic,
                    "kernel": head["kernel"], "flops_per_launch": runner.flops,
                    "ms_per_launch": head["ms_per_launch"],
                    "ms_per_launch_back_to_back": head["ms_per_launch_back_to_back"],
                    "peak_kind": f"bf16 dense burst ({peaks['source']})",
                    "peak_sustained": peaks["bf16_tflops_sustained"],
                    "frac_of_sustained": head["frac_of_sustained"]}
    append_in_step = dict(head["append"])
    append_in_step["traffic"] = recorded_traffic("append_uniform") if full_uniform else None

    e2e = None
    if not args.no_e2e:
        e2e_s, h2d, d2h, _ = time_e2e(runner, stream, args.e2e_steps, 1)
        e2e_s = max_over_ranks(e2e_s, dist_on, device)
        e2e = {"value": aggregate_value(runner.flops, e2e_s * 1e3, world), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": args.e2e_steps, "ms_per_step": e2e_s * 1e3}
    launches = runner.launches_per_step() * args.steps
    tokens = runner.tokens
    runner.close()
    del runner, stream
    torch.cuda.empty_cache()

    extra = {}
    if not args.no_extra and not args.seqs and args.workload == "uniform" and \
            args.kv_format == "nvfp4":
        for key, name, fmt in EXTRA:
            c2 = ClockSampler(local_rank)
            c2.start()
            r2, s2, t2 = measure(fi, name, device, args.extra_steps, 3, dist_on, kv_format=fmt)
            ck = c2.stop()
            e = attention_entry(r2, t2, peaks,
                                "decode_128x4096" if name == "decode" else None)
            e["workload"] = WORKLOAD_DESC[name] + (" [FP8 (E4M3) paged KV]" if fmt == "fp8" else "")
            e["steps"] = args.extra_steps
            e["clocks"] = {"sm_mhz": ck["sm_mhz"], "reasons": ck["reasons"]}
            extra[key] = e
            r2.close()
            del r2, s2
            torch.cuda.empty_cache()

    plan_us = None
    if not args.no_extra and rank == 0:
        plan_us = {"unit": "us per call", "what": "fi_prefill_plan / fi_decode_plan through the "
                   "Python binding, stream idle (H_q=32, H_kv=8, D=128, ps=16; uniform: "
                   "1024 tokens per sequence; ragged: log-uniform lengths in [128, 16384])",
                   **time_plan_host(fi, device)}

    app = None
    if not args.no_append_bench and rank == 0:
        a = time_append_cold(fi, device)
        app = {"workload": "append bandwidth: 8192 tokens, H_kv=8, head_dim=128, "
                           "page_size=16, 5% slots=-1, random page permutation",
               "gbs_cold_l2": a["bytes"] / (a["cold_ms"] * 1e-3) / 1e9,
               "gbs_warm_l2": a["bytes"] / (a["warm_ms"] * 1e-3) / 1e9,
               "us_cold_l2": a["cold_ms"] * 1e3, "us_warm_l2": a["warm_ms"] * 1e3,
               "algorithmic_bytes": a["bytes"],
               "frac_cold_l2": a["bytes"] / (a["cold_ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
               "traffic": recorded_traffic("append_8192"),
               "peak_gbs": peaks["hbm_gbs"],
               "cold_l2_method": f"{a['sets']} rotating buffer sets "
                                 f"({a['sets'] * a['set_bytes'] / 2**20:.0f} MiB) in one CUDA graph",
               "status": a["status"]}

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1 and args.kv_format == "nvfp4":
        r = oracle_sample(args.workload, seed=0)
        cpu = {"value": r["flops"] / (r["t_append"] + r["t_attn"]) / 1e12, "unit": UNIT,
               "cores": r["threads"], "kind": "oracle", "sample": r["desc"],
               "attention_only_tflops": r["flops"] / r["t_attn"] / 1e12}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[args.workload] +
                   (f" (first {args.seqs} sequences only)" if args.seqs else "") +
                   (" [FP8 (E4M3) paged KV variant]" if args.kv_format == "fp8" else ""),
                   "kv_format": args.kv_format,
                   "tokens": tokens,
                   "flops_per_step": head["flops_per_launch"],
                   "l2": "inputs larger than L2 (Q 8.6 GB, KV cache 1.2 GB per step)"
                   if args.workload == "uniform" and not args.seqs else "see workload",
                   "step": "plan (upload) -> append -> prefill, no event between the kernels",
                   "parallelism": f"replicas x{world} (independent shards, no collective)"},
        "roofline": roofline,
        "append_in_step": append_in_step,
        "workloads": extra or None,
        "append_bench": app,
        "plan_host_us": plan_us,
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": launches,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist_on:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
