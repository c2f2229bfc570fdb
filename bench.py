#!/usr/bin/env python
"""Benchmark of the speculative-decoding verification step on GB300.

One "step" is one full verification call (both phases: row statistics,
then accept scan + final draw) over one synthetic batch already resident in
HBM.  Default workload: c3 (B=64 sequences, k=5 drafts, V=151936, bf16
logits, T=1), 213.9 MB of logits per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c3]
    python bench.py --impl reference ...    # the fp64 CPU oracle, host cores

Prints one JSON line (rank 0).  value = logit GB/s (every logit read once),
the metric the verification step is quoted in; steps/s, logits/s and the
fraction of the measured HBM peak are reported beside it.

Timing: W untimed warm-up steps, then K steps bracketed by a barrier and
torch.cuda.synchronize() on both sides, CUDA events on the library's stream,
max over ranks.  The inputs (214 MB) exceed the 126 MB L2 and two copies
alternate between steps, so every step streams from HBM.  nvidia-smi clocks
are sampled during the timed region.  With N > 1 (torchrun) every rank runs
an independent replica on its own GPU (sequences are independent; there is
no data-path collective) and value is the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0
_CSRC = os.path.join(ROOT, "speculative_decoding_verification_top_gb300", "csrc")
_INCLUDE = os.path.join(ROOT, "include")


def include_closure(tu):
    """The translation unit `tu` and every file it reaches through
    `#include "..."` (looked up beside the including file, then in csrc/ and
    include/), in a fixed order: the unit first, then the rest sorted."""
    seen, todo = [], [os.path.abspath(tu)]
    while todo:
        f = todo.pop()
        if f in seen:
            continue
        seen.append(f)
        for name in re.findall(r'^\s*#\s*include\s+"([^"]+)"', open(f).read(), flags=re.M):
            for d in (os.path.dirname(f), _CSRC, _INCLUDE):
                cand = os.path.abspath(os.path.join(d, name))
                if os.path.exists(cand):
                    todo.append(cand)
                    break
            else:
                raise FileNotFoundError("%s includes %s, which was not found" % (f, name))
    return [seen[0]] + sorted(seen[1:])


# The committed ncu summary of each row-phase kernel, and the sources whose
# hash it was taken on: the kernel's translation unit and everything it
# includes (its traffic is reported only while they match).
PROFILES = {
    "stream_kernel": (os.path.join(ROOT, "profiles", "stream_kernel_c3.md"),
                      include_closure(os.path.join(_CSRC, "rows.cu"))),
    "topp_kernel": (os.path.join(ROOT, "profiles", "topp_kernel_c4.md"),
                    include_closure(os.path.join(_CSRC, "topp.cu"))),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="c3", choices=["c1", "c2", "c3", "c4", "c5"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="budget of the CPU-oracle baseline sample (each of one core, all cores)")
    ap.add_argument("--no-blocks", action="store_true",
                    help="only the headline workload (no c1/c2/c4/c5 blocks after it)")
    ap.add_argument("--quick", action="store_true",
                    help="a short run for profiling: no blocks, no load around the timed "
                         "calls, 50 individually timed calls")
    return ap.parse_args()


def make_workload(name):
    wl = workloads.CONFIGS[name]()
    mode = "tree" if name == "c5" else "stochastic"
    return wl, mode


def describe(wl, mode):
    if mode == "tree":
        return {"workload": "%s: greedy tree verification, B=%d, N=%d nodes, V=%d, %s logits"
                            % (wl.name, wl.B, wl.N, wl.V, wl.dtype),
                "B": wl.B, "N": wl.N, "V": wl.V, "dtype": wl.dtype}
    return {"workload": "%s: stochastic verification, B=%d, k=%d, V=%d, %s logits, T=%g, top_p=%g"
                        % (wl.name, wl.B, wl.k, wl.V, wl.dtype, wl.T, wl.top_p),
            "B": wl.B, "k": wl.k, "V": wl.V, "dtype": wl.dtype, "T": wl.T, "top_p": wl.top_p}


# ------------------------------------------------------------ distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms."""
    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append(dict(sm=float(parts[2]), smax=float(parts[3]), power=float(parts[4]),
                                 hw=parts[6], hwt=parts[7], swt=parts[8], cap=parts[9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("cap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median([r["sm"] for r in rows])),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "power_w_max": max(r["power"] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


# ------------------------------------------------------------------- peaks

def hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_code_hash(paths):
    """First 16 hex digits of the sha256 of the sources' code: comments,
    blank lines and trailing spaces removed, so that a comment edit does not
    count as a kernel change."""
    h = hashlib.sha256()
    for path in paths:
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for line in text.splitlines():
            line = re.sub(r"//.*$", "", line).rstrip()
            if line:
                h.update(line.encode() + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic(kernel, config):
    """dram bytes per launch of `kernel` from its committed ncu summary, if
    that was taken on this workload and on the current kernel code (else
    None)."""
    summary, sources = PROFILES[kernel]
    try:
        text = open(summary).read()
        src = source_code_hash(sources)
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if line.split(":", 1)[0] in ("traffic_bytes_per_launch", "source_code_sha256_16", "workload"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if (fields.get("source_code_sha256_16") != src or fields.get("workload") != config
            or "traffic_bytes_per_launch" not in fields):
        return None
    return float(fields["traffic_bytes_per_launch"])


# ---------------------------------------------------------------- our arm

def to_dev(a, dev):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


class Job:
    """Device buffers and bound launchers for one workload."""

    def __init__(self, wl, mode, dev):
        import torch
        import speculative_decoding_verification_top_gb300 as sv
        self.sv, self.wl, self.mode, self.dev = sv, wl, mode, dev
        self.stream = torch.cuda.current_stream(dev)
        self.sets = []
        if mode == "tree":
            base = (to_dev(wl.target, dev), to_dev(wl.parents, dev), to_dev(wl.node_tokens, dev))
            self.sets = [base, tuple(a.clone() for a in base)]
            W = wl.D + 1
            self.out_t = torch.empty((wl.B, W), dtype=torch.int32, device=dev)
            self.out_n = torch.empty((wl.B,), dtype=torch.int32, device=dev)
            self.out_p = torch.empty((wl.B, W), dtype=torch.int32, device=dev)
            nbytes = sv.spec_verify_tree_workspace_size(wl.B, wl.N, wl.V)
            self.launches_per_step = 2
        else:
            base = (to_dev(wl.target, dev), to_dev(wl.draft, dev), to_dev(wl.draft_tokens, dev),
                    to_dev(wl.uniforms, dev))
            self.sets = [base, tuple(a.clone() for a in base)]
            self.out_t = torch.empty((wl.B, wl.k + 1), dtype=torch.int32, device=dev)
            self.out_n = torch.empty((wl.B,), dtype=torch.int32, device=dev)
            nbytes = sv.spec_verify_workspace_size(wl.B, wl.k, wl.V)
            self.launches_per_step = 2
        self.ws = sv.new_workspace(nbytes, dev)
        self.dtype = sv.SPEC_BF16 if wl.dtype == workloads.BF16 else sv.SPEC_F32

    def chain_args(self, i):
        t, d, x, u = self.sets[i % 2]
        wl, sv = self.wl, self.sv
        return (t.data_ptr(), d.data_ptr(), x.data_ptr(), u.data_ptr(), wl.B, wl.k, wl.V, wl.T,
                wl.top_p, sv.SPEC_STOCHASTIC, self.dtype, self.out_t.data_ptr(),
                self.out_n.data_ptr(), self.ws.data_ptr(), self.ws.numel(),
                self.stream.cuda_stream)

    def step(self, i):
        sv = self.sv
        if self.mode == "tree":
            t, p, x = self.sets[i % 2]
            wl = self.wl
            sv.spec_verify_tree(t.data_ptr(), p.data_ptr(), x.data_ptr(), wl.B, wl.N, wl.V, wl.D,
                                self.dtype, self.out_t.data_ptr(), self.out_n.data_ptr(),
                                self.out_p.data_ptr(), self.ws.data_ptr(), self.ws.numel(),
                                self.stream.cuda_stream)
        else:
            sv.spec_verify_sample(*self.chain_args(i))

    def rows_only(self, i):
        """The row phase of one chain step alone."""
        self.sv.spec_verify_sample_rows(*self.chain_args(i))


def call_times_ms(launch, n, stream, chunk=100):
    """Device time of each launch(i), i < n, bracketed by CUDA events on
    `stream`.  Each chunk of launches is queued behind a ~25 ms device-side
    sleep, so the host is far ahead when they run: the events time the
    kernels back to back, not the host's launch latency."""
    import torch
    times = []
    for c0 in range(0, n, chunk):
        m = min(chunk, n - c0)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(m)]
        torch.cuda._sleep(50_000_000)
        for j, (a, b) in enumerate(evs):
            a.record(stream)
            launch(c0 + j)
            b.record(stream)
        torch.cuda.synchronize()
        times += [a.elapsed_time(b) for a, b in evs]
    return times


def device_launch_ms(launch, n, stream, chunk=100):
    """Mean of call_times_ms."""
    return float(np.mean(call_times_ms(launch, n, stream, chunk)))


def per_call(times_ms):
    """Best, median and mean of per-call device times, in microseconds."""
    t = np.asarray(times_ms) * 1e3
    return {"n": int(t.size), "best_us": round(float(t.min()), 2),
            "median_us": round(float(np.median(t)), 2), "mean_us": round(float(t.mean()), 2)}


def soak(job, seconds, step0=0):
    """Whole calls back to back for about `seconds` (untimed load that keeps
    the clocks where the timed calls run them)."""
    import torch
    if seconds <= 0:
        return step0
    t0, i = time.perf_counter(), step0
    while time.perf_counter() - t0 < seconds:
        for _ in range(50):
            job.step(i)
            i += 1
        torch.cuda.synchronize()
    return i


def pinned_h2d_gbs(dev, nbytes=256 << 20, reps=8):
    """Host-to-device copy rate from pinned memory: one large copy repeated,
    timed with CUDA events (the link's rate for the e2e leg's copies)."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        d.copy_(h, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    return round(nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)


def timed_device(job, steps, warmup, world, kernel_launches=500):
    """Whole verify calls back to back (nothing enqueued between them), then,
    for the roofline, the row kernel alone in launches bracketed by events."""
    import torch
    for i in range(warmup):
        job.step(i)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    ev0.record(job.stream)
    for i in range(steps):
        job.step(i)
    ev1.record(job.stream)
    torch.cuda.synchronize()
    barrier(world)
    total_ms = ev0.elapsed_time(ev1)
    rows_ms = None
    if job.mode != "tree":
        for i in range(3):
            job.rows_only(i)
        torch.cuda.synchronize()
        rows_ms = device_launch_ms(job.rows_only, min(steps, kernel_launches), job.stream)
        job.step(0)  # leave the workspace as a finished call left it
        torch.cuda.synchronize()
    return total_ms, rows_ms


def timed_acceptance(job, launches=200):
    """spec_verify_acceptance on the finished call's workspace: launches
    bracketed by events, alternating the two (identical) input copies so
    that consecutive launches do not find their rows in L2."""
    import torch
    wl, sv = job.wl, job.sv
    beta = torch.empty((wl.B, wl.k), dtype=torch.float32, device=job.dev)
    tv = torch.empty((wl.B, wl.k), dtype=torch.float32, device=job.dev)

    def one(i):
        t, d = job.sets[i % 2][:2]
        sv.spec_verify_acceptance(t.data_ptr(), d.data_ptr(), wl.B, wl.k, wl.V, wl.T, wl.top_p,
                                  0, job.dtype, beta.data_ptr(), tv.data_ptr(), job.ws.data_ptr(),
                                  job.ws.numel(), job.stream.cuda_stream)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    ms = device_launch_ms(one, launches, job.stream)
    esz = 2 if wl.dtype == workloads.BF16 else 4
    listed = wl.top_p < 1.0
    # Without top-p both rows of every pair are read once; with top-p the
    # pairs are summed over the nucleus lists (no row is read when every
    # list fits), so no byte count is claimed.
    nbytes = None if listed else 2 * wl.B * wl.k * wl.V * esz
    out = {"kernel": "accept_kernel", "launches": launches, "avg_launch_us": round(ms * 1e3, 2),
           "mean_beta": round(float(beta.double().mean().item()), 5),
           "path": "nucleus lists" if listed else "both rows streamed"}
    if nbytes:
        out["algorithmic_bytes"] = nbytes
        out["achieved_gbs"] = round(nbytes / (ms * 1e-3) / 1e9, 1)
    return out


def timed_probs(job, launches=200):
    """spec_verify_sample_probs on the same target logits with the draft
    given as fp32 probability rows (seeded synthetic rows, drawn once):
    device time per call.  Bytes counted: the k+1 target rows of every
    sequence, plus the fp32 draft row the final draw reads for each
    sequence that rejected (its residual)."""
    import torch
    wl, sv = job.wl, job.sv
    rng = np.random.default_rng(20240)
    q, toks = workloads.draft_prob_rows(rng, workloads.as_f32(wl.target), wl.k)
    qd, xd = to_dev(q, job.dev), to_dev(toks, job.dev)

    def one(i):
        t, _, _, u = job.sets[i % 2]
        sv.spec_verify_sample_probs(t.data_ptr(), qd.data_ptr(), xd.data_ptr(), u.data_ptr(),
                                    wl.B, wl.k, wl.V, wl.T, wl.top_p, 0, job.dtype,
                                    job.out_t.data_ptr(), job.out_n.data_ptr(),
                                    job.ws.data_ptr(), job.ws.numel(), job.stream.cuda_stream)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    ms = device_launch_ms(one, launches, job.stream)
    n = job.out_n.cpu().numpy()
    esz = 2 if wl.dtype == workloads.BF16 else 4
    nbytes = wl.B * (wl.k + 1) * wl.V * esz + int(((n >= 0) & (n < wl.k)).sum()) * wl.V * 4
    job.step(0)  # leave the workspace as a logits call left it
    torch.cuda.synchronize()
    return {"entry": "spec_verify_sample_probs", "launches": launches,
            "avg_call_us": round(ms * 1e3, 2), "bytes": nbytes,
            "achieved_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "accepted_hist": np.bincount(np.maximum(n, 0), minlength=wl.k + 1).tolist()}


def timed_tree_mask(job, launches=200):
    """spec_verify_tree_mask: the workload's tree for each of its B
    sequences, and a large case (64 complete 4-ary trees of 1024 nodes,
    depth 5); mask and positions; device time per call and the bytes
    written."""
    import torch
    wl, sv = job.wl, job.sv
    out = {}
    big = np.broadcast_to(((np.arange(1024) - 1) // 4).astype(np.int32), (64, 1024)).copy()
    big[:, 0] = -1
    cases = [("workload", np.broadcast_to(wl.parents, (wl.B, wl.N)).copy()), ("B64_N1024", big)]
    for name, par in cases:
        B, N = par.shape
        p = to_dev(par, job.dev)
        mask = torch.empty((B, N, N), dtype=torch.uint8, device=job.dev)
        pos = torch.empty((B, N), dtype=torch.int32, device=job.dev)

        def one(i):
            sv.spec_verify_tree_mask(p.data_ptr(), None, B, N, mask.data_ptr(), None,
                                     pos.data_ptr(), job.stream.cuda_stream)

        for i in range(3):
            one(i)
        torch.cuda.synchronize()
        ms = device_launch_ms(one, launches, job.stream)
        nbytes = B * N * N + 4 * B * N + 4 * B * N  # mask + positions written, parents read
        out[name] = {"B": B, "N": N, "avg_call_us": round(ms * 1e3, 2), "bytes": nbytes,
                     "achieved_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    return out


def timed_topk(job, K=50, launches=200):
    """spec_verify_sample_topk with top-k K on the workload (and its top-p):
    device time per call over the same logits."""
    import torch
    wl, sv = job.wl, job.sv

    def one(i):
        a = job.chain_args(i)
        sv.spec_verify_sample_topk(*a[:9], K, *a[9:])

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    ms = device_launch_ms(one, launches, job.stream)
    nbytes = wl.logit_bytes()
    job.step(0)  # leave the workspace as a plain call left it
    torch.cuda.synchronize()
    return {"entry": "spec_verify_sample_topk", "top_k": K, "top_p": wl.top_p,
            "launches": launches, "avg_call_us": round(ms * 1e3, 2), "bytes": nbytes,
            "achieved_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}


def timed_tree_sample(job, launches=100):
    """spec_verify_tree_sample on c5's tree shape, sampled (draft rows =
    target + noise, children drawn from their parent's draft row): device
    time per call."""
    import torch
    sv = job.sv
    tr = workloads.c5s(B=job.wl.B, V=job.wl.V)
    dt = sv.SPEC_BF16 if tr.dtype == workloads.BF16 else sv.SPEC_F32
    tg, dr = to_dev(tr.target, job.dev), to_dev(tr.draft, job.dev)
    par, tok = to_dev(tr.parents, job.dev), to_dev(tr.node_tokens, job.dev)
    uni = to_dev(tr.uniforms, job.dev)
    W = tr.D + 1
    ot = torch.empty((tr.B, W), dtype=torch.int32, device=job.dev)
    on = torch.empty((tr.B,), dtype=torch.int32, device=job.dev)
    op = torch.empty((tr.B, W), dtype=torch.int32, device=job.dev)
    ws = sv.new_workspace(sv.spec_verify_tree_sample_workspace_size(tr.B, tr.N, tr.V), job.dev)

    def one(i):
        sv.spec_verify_tree_sample(tg.data_ptr(), dr.data_ptr(), par.data_ptr(), tok.data_ptr(),
                                   uni.data_ptr(), tr.B, tr.N, tr.V, tr.D, tr.T, 1.0, 0, dt,
                                   ot.data_ptr(), on.data_ptr(), op.data_ptr(), ws.data_ptr(),
                                   ws.numel(), job.stream.cuda_stream)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    ms = device_launch_ms(one, launches, job.stream)
    depths = np.bincount(np.maximum(on.cpu().numpy(), 0), minlength=W).tolist()
    nbytes = tr.logit_bytes()
    return {"entry": "spec_verify_tree_sample", "B": tr.B, "N": tr.N, "V": tr.V,
            "avg_call_us": round(ms * 1e3, 2), "bytes_rows": nbytes,
            "achieved_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "depth_hist": depths}


def timed_e2e(job, steps):
    """Host buffers -> device -> library call -> results back to the host,
    every step.  Two device input sets alternate: the copy of step i+1 (its
    own stream) overlaps the call and the read-back of step i; a copy into a
    set waits until the call that last read it has finished."""
    import torch
    wl = job.wl
    def pinned(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:  # bf16 bit patterns
            a = a.view(np.int16)
        return torch.from_numpy(a).pin_memory()

    if job.mode == "tree":
        host_in = [pinned(a) for a in (wl.target, wl.parents, wl.node_tokens)]
        outs = (job.out_t, job.out_n, job.out_p)
    else:
        host_in = [pinned(a) for a in (wl.target, wl.draft, wl.draft_tokens, wl.uniforms)]
        outs = (job.out_t, job.out_n)
    host_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    views = [[d.view(torch.int16) if d.dtype == torch.bfloat16 else d for d in job.sets[j]]
             for j in range(2)]
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = sum(h.numel() * h.element_size() for h in host_out)
    copy_stream = torch.cuda.Stream(device=job.dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    for e in done:
        e.record(job.stream)

    def one(i):
        j = i % 2
        copy_stream.wait_event(done[j])
        with torch.cuda.stream(copy_stream):
            for h, d in zip(host_in, views[j]):
                d.copy_(h, non_blocking=True)
        copied[j].record(copy_stream)
        job.stream.wait_event(copied[j])
        job.step(j)
        for h, o in zip(host_out, outs):
            h.copy_(o, non_blocking=True)
        done[j].record(job.stream)

    for i in range(4):
        one(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(job.stream)
    copy_stream.wait_event(e0)
    for i in range(steps):
        one(i)
    e1.record(job.stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    return e0.elapsed_time(e1), wall * 1e3, h2d, d2h


def _oracle_sequence(arrs, mode, b, meta):
    """One whole sequence b of a workload through the fp64 oracle; returns
    the logit bytes it read."""
    import oracle
    sl = slice(b, b + 1)
    if mode == "tree":
        oracle.verify_tree(arrs["target"][sl], arrs["parents"], arrs["node_tokens"][sl], meta["D"])
    else:
        oracle.verify_sample(arrs["target"][sl], arrs["draft"][sl], arrs["draft_tokens"][sl],
                             arrs["uniforms"][sl], T=meta["T"], top_p=meta["top_p"])
    return meta["bytes_per_seq"]


def _oracle_worker(task):
    """A spawned worker: sequences b0, b0+1, ... (mod B), n of them, from
    the workload's arrays memory-mapped from `folder`."""
    folder, mode, meta, b0, n = task
    arrs = {k: np.load(os.path.join(folder, k + ".npy"), mmap_mode="r") for k in meta["arrays"]}
    done = 0
    for i in range(n):
        done += _oracle_sequence(arrs, mode, (b0 + i) % meta["B"], meta)
    return done


def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(wl, mode, seconds, all_cores=True):
    """The fp64 oracle, as it stands, on the host cores over bounded
    samples of the same workload: whole sequences, round-robin over the
    batch.  First one core for `seconds`; then, if all_cores, every core at
    once (one spawned process per core, each running sequences from the
    workload's arrays memory-mapped from a temporary folder) for about
    `seconds` more."""
    import oracle
    oracle.build()
    if mode == "tree":
        arrs = {"target": wl.target, "parents": wl.parents, "node_tokens": wl.node_tokens}
        meta = {"D": wl.D, "bytes_per_seq": wl.logit_bytes() // wl.B}
    else:
        arrs = {"target": wl.target, "draft": wl.draft, "draft_tokens": wl.draft_tokens,
                "uniforms": wl.uniforms}
        meta = {"T": wl.T, "top_p": wl.top_p, "bytes_per_seq": wl.logit_bytes() // wl.B}
    meta.update(B=wl.B, arrays=sorted(arrs))
    done, bytes_done, t0 = 0, 0, time.perf_counter()
    while True:
        bytes_done += _oracle_sequence(arrs, mode, done % wl.B, meta)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    one = {"value": bytes_done / el / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": "%d whole sequences of %s (round-robin over the batch), %.1f s on one core"
                     % (done, wl.name, el)}
    cores = _host_cores()
    if not all_cores or cores < 2:
        return dict(one, host_cores=cores)
    import multiprocessing as mp
    per = max(1, int(round(done / el * seconds)))  # sequences per worker, about `seconds`
    with tempfile.TemporaryDirectory() as folder:
        for k, v in arrs.items():
            np.save(os.path.join(folder, k + ".npy"), np.ascontiguousarray(v))
        ctx = mp.get_context("spawn")
        with ctx.Pool(cores) as pool:
            pool.map(_oracle_worker, [(folder, mode, meta, w, 1) for w in range(cores)])  # start-up
            t0 = time.perf_counter()
            got = pool.map(_oracle_worker, [(folder, mode, meta, w * per, per)
                                            for w in range(cores)])
            el2 = time.perf_counter() - t0
    # the baseline: every core; the one-core sample beside it
    return {"value": sum(got) / el2 / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "%d whole sequences of %s, %d per process on %d processes (one per core), "
                      "%.1f s" % (per * cores, wl.name, per, cores, el2),
            "host_cores": cores, "one_core": one}


def chain_block(name, dev, peak, cpu_seconds, calls=100):
    """Another chain workload, measured after the headline: best/median/mean
    of `calls` whole calls and of the row-phase kernel alone, the roofline of
    that kernel, and the one-core oracle on a bounded sample."""
    import torch
    wl, mode = make_workload(name)
    job = Job(wl, mode, dev)
    for i in range(3):
        job.step(i)
    torch.cuda.synchronize()
    calls_t = per_call(call_times_ms(job.step, calls, job.stream))
    rows_t = per_call(call_times_ms(job.rows_only, calls, job.stream))
    job.step(0)
    torch.cuda.synchronize()
    nbytes = wl.logit_bytes(mode)
    kern = "topp_kernel" if wl.top_p < 1.0 else "stream_kernel"
    rows_gbs = nbytes / (rows_t["mean_us"] * 1e-6) / 1e9
    call_gbs = nbytes / (calls_t["median_us"] * 1e-6) / 1e9
    out = {"workload": describe(wl, mode)["workload"], "logit_bytes": nbytes,
           "inputs_vs_l2": "two input copies of %.1f MB alternate between calls (L2: 126 MB)"
                           % (nbytes / 1e6),
           "ms_per_call": round(calls_t["median_us"] * 1e-3, 5), "calls": calls_t,
           "gbs": round(call_gbs, 1), "frac": round(call_gbs / peak, 4),
           "verify_calls_per_s": round(1e6 / calls_t["median_us"], 1),
           "roofline": {"bound": "hbm", "kernel": kern, "avg_launch_us": rows_t["mean_us"],
                        "launch": rows_t, "achieved": round(rows_gbs, 1), "peak": peak,
                        "unit": "GB/s", "frac": round(rows_gbs / peak, 4),
                        "traffic": profiled_traffic(kern, name), "algorithmic_bytes": nbytes},
           "cpu_baseline": cpu_baseline(wl, mode, cpu_seconds, all_cores=False)}
    del job
    torch.cuda.empty_cache()
    return out


def tree_block(dev, peak, cpu_seconds, calls=100):
    """c5 (greedy tree), with the stochastic tree (on c5's shape) and the
    tree mask beside it."""
    import torch
    wl, mode = make_workload("c5")
    job = Job(wl, mode, dev)
    for i in range(3):
        job.step(i)
    torch.cuda.synchronize()
    calls_t = per_call(call_times_ms(job.step, calls, job.stream))
    nbytes = wl.logit_bytes(mode)
    gbs = nbytes / (calls_t["median_us"] * 1e-6) / 1e9
    out = {"workload": describe(wl, mode)["workload"], "logit_bytes": nbytes,
           "ms_per_call": round(calls_t["median_us"] * 1e-3, 5), "calls": calls_t,
           "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
           "roofline": {"bound": "hbm", "kernel": "stream_kernel+tree_kernel",
                        "avg_launch_us": calls_t["mean_us"], "achieved": round(gbs, 1),
                        "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
                        "traffic": None, "algorithmic_bytes": nbytes},
           "cpu_baseline": cpu_baseline(wl, mode, cpu_seconds, all_cores=False)}
    ts = timed_tree_sample(job)
    ts["frac"] = round(ts["achieved_gbs"] / peak, 4)
    out["tree_sample"] = ts
    out["tree_mask"] = timed_tree_mask(job)
    del job
    torch.cuda.empty_cache()
    return out


def c1_block(dev, calls=200):
    """c1 (B=1, k=3, V=32, fp32): the latency of one call; and its batched
    form (10^5 replicated steps in one call): sequence steps per second."""
    import torch
    out = {}
    for label, steps in (("B1_latency", 1), ("B100000", 100_000)):
        wl = workloads.c1(steps=steps)
        job = Job(wl, "stochastic", dev)
        for i in range(3):
            job.step(i)
        torch.cuda.synchronize()
        t = per_call(call_times_ms(job.step, calls if steps == 1 else 50, job.stream))
        out[label] = {"B": wl.B, "k": wl.k, "V": wl.V, "calls": t,
                      "sequence_steps_per_s": round(wl.B * 1e6 / t["median_us"], 1)}
        del job
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    import speculative_decoding_verification_top_gb300 as sv
    world, rank, local = dist_setup()
    sv.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl, mode = make_workload(args.config)
    job = Job(wl, mode, dev)
    job.step(0)
    torch.cuda.synchronize()

    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = visible.split(",")[local] if visible else str(local)
    clocks = ClockSampler(smi_index)
    time.sleep(0.3)
    # The sampler polls every 20 ms: untimed calls before and after the
    # timed ones keep the GPU under the same load for ~1 s around them.
    nxt = soak(job, 0.0 if args.quick else 0.6)
    total_ms, rows_ms = timed_device(job, args.steps, args.warmup, world)
    soak(job, 0.0 if args.quick else 0.4, nxt)
    clk = clocks.stop()
    if clk is not None:
        clk["window"] = ("the timed calls plus ~1 s of the same calls around them "
                         "(20 ms sampling)")
    # best / median / mean of individually timed calls (inputs alternate
    # between two copies larger than L2)
    calls = per_call(call_times_ms(job.step, 50 if args.quick else max(args.steps, 200),
                                   job.stream))
    accept = timed_acceptance(job) if mode != "tree" else None
    probs = timed_probs(job) if mode != "tree" else None
    topk = timed_topk(job) if mode != "tree" else None
    tmask = timed_tree_mask(job) if mode == "tree" else None
    tsample = timed_tree_sample(job) if mode == "tree" else None
    total_ms = max_over_ranks(total_ms, world)

    nbytes = wl.logit_bytes(mode)
    ms_step = total_ms / args.steps
    value = world * nbytes * args.steps / (total_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    e2e_ms, e2e_wall_ms, h2d, d2h = timed_e2e(job, args.e2e_steps)
    h2d_peak = pinned_h2d_gbs(dev)
    e2e_ms = max_over_ranks(e2e_ms, world)
    e2e_value = world * nbytes * args.e2e_steps / (e2e_ms * 1e-3) / 1e9

    if rows_ms is not None:
        # The row phase: one stream_kernel launch, or with top-p one
        # topp_kernel launch.
        kern = "topp_kernel" if wl.top_p < 1.0 else "stream_kernel"
        achieved = nbytes / (rows_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": kern,
                    "achieved": round(achieved, 1),
                    "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                    "frac": round(achieved / peak, 4),
                    "traffic": profiled_traffic(kern, args.config),
                    "algorithmic_bytes": nbytes, "avg_launch_us": round(rows_ms * 1e3, 2)}
    else:
        per_launch_ms = ms_step  # the tree call: argmax rows kernel dominates
        achieved = nbytes / (per_launch_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": "stream_kernel+tree_kernel", "achieved": round(achieved, 1),
                    "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "traffic": None,
                    "algorithmic_bytes": nbytes, "avg_launch_us": round(per_launch_ms * 1e3, 2)}

    out = {
        "metric": "verify logits GB/s (% of GB300 HBM peak) and verify steps/sec at (B,k,V)",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "impl": "ours",
        "config": describe(wl, mode),
        "inputs_vs_l2": ("inputs %d MB > 126 MB L2; two input copies alternate between steps"
                         % (nbytes // 10**6)),
        "calls": calls,
        "frac_of_peak": round(value / world / peak, 4), "peak_gbs": peak, "peak_kind": peak_kind,
        "frac_of_nominal_8tbs": round(value / world / 8000.0, 4),
        "verify_calls_per_s": round(world * args.steps / (total_ms * 1e-3), 1),
        "sequence_steps_per_s": round(world * wl.B * args.steps / (total_ms * 1e-3), 1),
        "logits_per_s": round(value * 1e9 / (2 if wl.dtype == workloads.BF16 else 4), 1),
        "roofline": roofline,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "steps": args.e2e_steps,
                "ms_per_step": round(e2e_ms / args.e2e_steps, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "h2d_pinned_gbs": h2d_peak,
                "h2d_pinned_note": "one 256 MiB pinned host-to-device copy, repeated, timed "
                                   "with CUDA events: the link rate the e2e copies share"},
        "gpu_launches": job.launches_per_step * args.steps,
        "clocks": clk,
    }
    if accept is not None:
        if "achieved_gbs" in accept:
            accept["frac"] = round(accept["achieved_gbs"] / peak, 4)
        out["acceptance"] = accept
    if tmask is not None:
        out["tree_mask"] = tmask
    if tsample is not None:
        out["tree_sample"] = tsample
    if topk is not None:
        topk["frac"] = round(topk["achieved_gbs"] / peak, 4)
        out["top_k"] = topk
    if probs is not None:
        probs["frac"] = round(probs["achieved_gbs"] / peak, 4)
        out["draft_probs"] = probs
    if rank == 0 and world == 1:
        out["cpu_baseline"] = cpu_baseline(wl, mode, args.cpu_seconds)
    if rank == 0 and world == 1 and args.config == "c3" and not (args.no_blocks or args.quick):
        # the other workloads, one block each (their own calls, after the
        # headline's timed region)
        cs = min(3.0, args.cpu_seconds)
        out["configs"] = {"c4": chain_block("c4", dev, peak, cs),
                          "c2": chain_block("c2", dev, peak, cs),
                          "c5": tree_block(dev, peak, cs),
                          "c1": c1_block(dev)}
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_reference(args):
    world, rank, _ = (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0)
    if rank != 0:
        return
    import oracle
    oracle.build()
    wl, mode = make_workload(args.config)
    per_seq = wl.logit_bytes(mode) // wl.B

    def one(i):
        sl = slice(i % wl.B, i % wl.B + 1)
        if mode == "tree":
            oracle.verify_tree(wl.target[sl], wl.parents, wl.node_tokens[sl], wl.D)
        else:
            oracle.verify_sample(wl.target[sl], wl.draft[sl], wl.draft_tokens[sl],
                                 wl.uniforms[sl], T=wl.T, top_p=wl.top_p)

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i)
    el = time.perf_counter() - t0
    value = per_seq * args.steps / el / 1e9
    sample = ("each step: one whole sequence of %s (round-robin over the batch) through the "
              "fp64 CPU oracle, one core" % wl.name)
    out = {
        "metric": "verify logits GB/s (% of GB300 HBM peak) and verify steps/sec at (B,k,V)",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference", "config": describe(wl, mode),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
