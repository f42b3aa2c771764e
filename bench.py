"""Benchmark: aggregated gradient GB/s on one GB300 and its fraction of the
HBM roofline, with the CPU oracle as the baseline.

The timed step (the line's `value`) is the largest single-GPU
configuration: Random SkipReduce on N = 8 ranks x M = 143,667,240 bf16 (a
VGG-19-sized flat gradient, N(0, 1e-2) cast to bf16) at skip fractions 0,
1/4 and 1/2, i.e. k = 0, 2 and 4 Reduce-Scatter steps skipped, one launch
each, in place, seed 0, iteration count = the step number.  Algorithmic
("roofline") bytes of a launch: (N - k) * M * 2 read + N * M * 2 written.
GB/s = those bytes / device time; the roofline fraction divides by the
measured HBM copy bandwidth.

Every other configuration is timed in the same run, after the step, as a
`part` with its bytes, median ms, GB/s and fraction: the N = 4, M = 2^20
fp32 ring (C1), the ResNet-50-sized fp32 ring and SkipReduce (C2), the C4
embedding-gradient union and push-side partition, the DGC top-5 % union
(C5b), the dense fp32 sweep N x M (C5a) and the next-row kernels
(AllReduce_Dropout, selective SkipReduce, Reduce-Scatter only, hash bitmap
encode / decode / index sets, group densification).  A configuration whose
inputs are smaller than twice the 129 MB L2 is timed over enough copies of
its buffers (used in turn) that every launch reads HBM; the tiniest sweep
points are latency-bound and flagged.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       [--parts all|none|PREFIX[,PREFIX...]] [--no-e2e] [--no-cpu-baseline]
With N > 1 (torchrun) every rank runs an independent replica of the whole
workload on its own GPU (the path has no exchange between GPUs: replicas
only); value = bytes of all ranks / the slowest rank's time.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "aggregated gradient GB/s at 1 GB300 and % of HBM roofline, vs host-oracle"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1000 * 1000
WORKLOAD = ("C3 dense SkipReduce N=8 M=143,667,240 bf16 (VGG-19-sized), Random SkipReduce at "
            "skip fractions 0, 1/4, 1/2 (k = 0, 2, 4), one in-place launch each per step")

# DRAM traffic of the dominant kernel from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum per launch), valid only while the kernel source is the
# one that was profiled.
TRAFFIC = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum on the C3 k = 0
    # launch: 2,298,799,872 B read + 2,239,374,848 B written (the rest of the
    # writes are still in L2 when the launch ends).
    "ring_fused_kernel<bf16>": {
        "source_sha256": "fb2c78050bb704767bc03b13c70c4983f16c37c746a451036e7291b8e04d9763",
        "bytes_per_launch": 4_538_174_720},
}

# Kernels of this library each call launches (counted from the library
# source; the status-word memsets of the sparse paths are runtime memsets,
# not counted).
LAUNCHES = {"ring": 1, "skip": 1, "rs_only": 1, "dropout": 1, "buckets": 1, "union": 5,
            "partition": 1, "hb_directory": 2, "hb_encode": 2, "hb_decode": 3, "hb_sets": 1,
            "densify": 2}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--parts", default="all",
                    help="the other configurations timed after the step: all, none, or "
                         "comma-separated name prefixes (c1, c2, c4, c5a, c5b, next)")
    ap.add_argument("--parts-only", action="store_true",
                    help="profiling: time only the selected parts (no step, no benchmark "
                         "line; prints one profiling line)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


# ---------------------------------------------------------------- timing
def max_over_ranks(ms, dist_mod, device):
    """The slowest rank's time (all_reduce MAX; a timing collective only)."""
    import torch

    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def job_throughput(step_bytes, steps, world, max_ms):
    """Whole-job GB/s: every replica processed step_bytes per step."""
    return world * step_bytes * steps / (max_ms / 1e3) / 1e9


def rotation_sets(set_bytes, cap=2048):
    """Copies of a configuration's buffers to use in turn so that their total
    exceeds twice the L2 (every launch then reads HBM): one when a copy
    alone does; capped, the capped case reported as L2-resident."""
    if set_bytes >= 2 * L2_BYTES:
        return 1, False
    need = -(-2 * L2_BYTES // max(1, set_bytes)) + 1
    return max(1, min(cap, need)), need > cap


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 200 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=5)
        return summarize_clocks(self.lines)


def summarize_clocks(lines):
    sm, mx, reasons = [], [], set()
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    for ln in lines:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            mx.append(float(parts[2]))
        except ValueError:
            continue
        for name, v in zip(names, parts[5:9]):
            if v.lower() == "active":
                reasons.add(name)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
            "samples": len(sm)}


# ---------------------------------------------------------------- the step
C3_KS = (0, 2, 4)


class Step:
    """The timed step's device buffers: the C3 bf16 rank buffers."""

    def __init__(self, torch, zr, dev):
        import numpy as np

        import workloads

        c = workloads.DENSE_C3
        self.torch, self.zr, self.dev = torch, zr, dev
        self.n, self.m = c["n"], c["m"]
        self.host = workloads.dense_c3()  # uint16 bf16 bit patterns, (n, m)
        h = torch.from_numpy(self.host.view(np.int16))
        self.dense = h.to(dev).view(torch.bfloat16)
        self.bufs = [self.dense[r] for r in range(self.n)]

    def launch_bytes(self, k):
        return (self.n - k) * self.m * 2 + self.n * self.m * 2

    def bytes(self):
        return sum(self.launch_bytes(k) for k in C3_KS)

    def run(self, i, events=None, bufs=None):
        zr = self.zr
        for k in C3_KS:
            zr.skipreduce(bufs or self.bufs, k=k, mode=zr.ZR_SKIP_RANDOM, seed=0, step=i)
            if events is not None:
                events[k].record()


def timed_step(torch, S, steps, warmup):
    """Device time of `steps` steps (CUDA events on the launching stream),
    and each launch's own duration per k."""
    for i in range(warmup):
        S.run(i)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    evs = [{k: torch.cuda.Event(enable_timing=True) for k in C3_KS} for _ in range(steps)]
    start.record()
    for i in range(steps):
        S.run(warmup + i, evs[i])
    torch.cuda.synchronize()
    total = start.elapsed_time(evs[-1][C3_KS[-1]])
    per = {k: [] for k in C3_KS}
    prev = start
    for e in evs:
        for k in C3_KS:
            per[k].append(prev.elapsed_time(e[k]))
            prev = e[k]
    return total, per


def timed_e2e(torch, S, steps):
    """The step through the public API from pinned host buffers: every step
    copies the 8 rank buffers host->device, runs the three SkipReduce calls
    and reads rank 0's result back.  Steps are pipelined over two device
    buffer slots and three streams (copy in, compute, copy out); a slot is
    refilled only after its last copy-out has finished."""
    import numpy as np

    h_in = torch.from_numpy(S.host.view(np.int16)).pin_memory()
    out = torch.empty(S.m, dtype=torch.int16).pin_memory()
    slots = [S.dense, torch.empty_like(S.dense)]
    h2d = h_in.numel() * 2
    d2h = S.m * 2
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def run(first, count):
        done = {}
        for i in range(first, first + count):
            d = slots[i % 2]
            bufs = [d[r] for r in range(S.n)]
            ev_in, ev_comp, ev_out = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
            with torch.cuda.stream(s_in):
                if i - 2 in done:
                    s_in.wait_event(done[i - 2])
                d.view(torch.int16).copy_(h_in, non_blocking=True)
                ev_in.record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in)
                S.run(i, bufs=bufs)
                ev_comp.record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp)
                out.copy_(d[0].view(torch.int16), non_blocking=True)
                ev_out.record(s_out)
            done[i] = ev_out
        return done

    run(0, 2)  # warm both slots
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    run(2, steps)
    t1.record(s_out)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    got = torch.from_numpy(out.numpy().view(np.int16)).view(torch.bfloat16).float()
    assert bool(torch.isfinite(got[:1000]).all())
    del slots[1]
    return ms, h2d, d2h


# ---------------------------------------------------------------- parts
def time_calls(torch, calls, steps, warmup, graph=False):
    """Median per-call device time (ms) of a list of calls used in turn (one
    per copy of a configuration's buffers): each round runs every call once;
    the round's time / len(calls) is one sample.  With graph=True the round
    is captured in a CUDA graph and replayed (small launches are then timed
    without the host's launch path)."""
    for i in range(warmup):
        for f in calls:
            f(i)
    torch.cuda.synchronize()
    run = None
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for f in calls:
                f(0)
        run = g.replay
        run()
        torch.cuda.synchronize()
    # back to back: an event after every round, no synchronisation between
    # rounds, so the device queue stays full
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    evs[0].record()
    for i in range(steps):
        if run is not None:
            run()
        else:
            for f in calls:
                f(warmup + i)
        evs[i + 1].record()
    torch.cuda.synchronize()
    times = [evs[i].elapsed_time(evs[i + 1]) / len(calls) for i in range(steps)]
    return statistics.median(times)


def part_entry(nbytes, ms, peak, **extra):
    gbs = nbytes / (ms / 1e3) / 1e9
    d = {"bytes": nbytes, "median_ms": ms, "gbs": gbs, "frac": gbs / peak}
    d.update(extra)
    return d


def wanted(sel, name):
    """Part `name` is selected (a prefix of it is), or, for a group prefix
    such as "c4", some part under it is."""
    if sel == "all":
        return True
    if sel == "none":
        return False
    return any(name.startswith(p) or p.startswith(name) for p in sel.split(","))


def run_parts(torch, zr, dev, sel, steps, warmup, peak, clock_off):
    """Every configuration other than the step, one after another; returns
    (parts, kernel launches made)."""
    import numpy as np

    import workloads

    parts = {}
    launches = 0

    def free():
        torch.cuda.synchronize()
        torch.cuda.empty_cache()

    # ---- C1: ring all-reduce, N = 4, M = 2^20 fp32, average (copies in turn)
    if wanted(sel, "c1_ring"):
        c = workloads.DENSE_C1
        n, m = c["n"], c["m"]
        base = torch.from_numpy(workloads.dense_c1()).to(dev)
        sets, resident = rotation_sets(n * m * 4)
        copies = [base.clone() for _ in range(sets)]
        calls = [(lambda i, x=x: zr.ring_allreduce([x[r] for r in range(n)], average=True))
                 for x in copies]
        ms = time_calls(torch, calls, steps, warmup, graph=True)
        parts["c1_ring"] = part_entry(2 * n * m * 4, ms, peak, n=n, m=m, dtype="f32",
                                      buffer_sets=sets, l2_resident=resident)
        launches += (steps + warmup + 1) * sets
        del base, copies, calls
        free()

    # ---- C2: ResNet-50-sized fp32 ring, SkipReduce and the next-row variants
    if wanted(sel, "c2_") or wanted(sel, "next_c2"):
        c = workloads.DENSE_C2
        n, m, k = c["n"], c["m"], c["skip_k"]
        x = torch.from_numpy(workloads.dense_c2()).to(dev)
        bufs = [x[r] for r in range(n)]
        items = [("c2_ring", lambda i: zr.ring_allreduce(bufs, average=True),
                  2 * n * m * 4, "ring"),
                 ("c2_skip_k4", lambda i: zr.skipreduce(bufs, k=k, mode=zr.ZR_SKIP_RANDOM,
                                                        seed=c["skip_seed"], step=i),
                  (2 * n - k) * m * 4, "skip")]
        if wanted(sel, "next_c2"):
            bucket = 25 * (1 << 20) // 4
            bks = []
            for b, lo in enumerate(range(0, m, bucket)):
                hi = min(lo + bucket, m)
                bks.append(dict(bufs=[x[r, lo:hi] for r in range(n)], k=0 if b == 0 else k,
                                mode=zr.ZR_SKIP_RANDOM, seed=b, step=0, m=hi - lo))
            b_bytes = sum((n - b["k"]) * b["m"] * 4 + n * b["m"] * 4 for b in bks)
            items += [
                ("next_c2_rs_only_k4", lambda i: zr.skipreduce(bufs, k=k, mode=zr.ZR_SKIP_RANDOM,
                                                               seed=0, step=i, rs_only=True),
                 (n - k) * m * 4 + m * 4, "rs_only"),
                ("next_c2_dropout_p50", lambda i: zr.allreduce_dropout(bufs, 0.5, seed=0, step=i),
                 2 * n * m * 4, "dropout"),
                ("next_c2_buckets", lambda i: zr.skipreduce_buckets(
                    [{kk: v for kk, v in dict(bb, step=i).items() if kk != "m"} for bb in bks]),
                 b_bytes, "buckets"),
            ]
        for name, fn, nbytes, kind in items:
            if not wanted(sel, name):
                continue
            ms = time_calls(torch, [fn], steps, warmup)
            parts[name] = part_entry(nbytes, ms, peak, n=n, m=m, dtype="f32")
            launches += (steps + warmup) * LAUNCHES[kind]
        del x, bufs, items
        free()

    # ---- C4: embedding-gradient union and push-side partition, densification,
    #      hash bitmaps (copies of the lists in turn where they fit in L2)
    if wanted(sel, "c4_") or wanted(sel, "next_c4"):
        c = workloads.SPARSE_C4
        m, P, seed = c["m"], c["n_parts"], c["part_seed"]
        idx_l, val_l = workloads.sparse_c4()
        n = len(idx_l)
        nnz = [a.size for a in idx_l]
        in_bytes = sum(nnz) * 8
        sets, resident = rotation_sets(in_bytes)
        d_sets = []
        for s in range(sets):
            di = [torch.from_numpy(a).to(dev) for a in idx_l]
            dv = [torch.from_numpy(v).to(dev) for v in val_l]
            d_sets.append((di, dv, zr.SparseWorkspace(n, m, P, sum(nnz), dev)))
        zr.sparse_aggregate(d_sets[0][0], d_sets[0][1], m, P, seed, work=d_sets[0][2])
        torch.cuda.synchronize()
        union = int(d_sets[0][2].out_nnz.item())
        if wanted(sel, "c4_union"):
            calls = [(lambda i, s=s: zr.sparse_aggregate(s[0], s[1], m, P, seed, work=s[2]))
                     for s in d_sets]
            ms = time_calls(torch, calls, steps, warmup, graph=True)
            parts["c4_union"] = part_entry(in_bytes + union * 8 + (P + 1) * 8 + 8, ms, peak,
                                           n=n, m=m, union=union, n_parts=P, buffer_sets=sets,
                                           l2_resident=resident,
                                           launches_per_call=LAUNCHES["union"])
            launches += (steps + warmup + 1) * sets * LAUNCHES["union"]
        if wanted(sel, "c4_partition"):
            p_out = [(torch.empty(nnz[0], dtype=torch.int32, device=dev),
                      torch.empty(nnz[0], dtype=torch.float32, device=dev),
                      torch.empty(P + 1, dtype=torch.int64, device=dev),
                      torch.empty(zr.zr_partition_workspace_size(nnz[0], P), dtype=torch.uint8,
                                  device=dev)) for _ in range(sets)]
            calls = [(lambda i, s=s, o=o: zr.partition(s[0][0], s[1][0], P, seed, o[0], o[1], o[2],
                                                        o[3])) for s, o in zip(d_sets, p_out)]
            ms = time_calls(torch, calls, steps, warmup, graph=True)
            parts["c4_partition"] = part_entry(nnz[0] * 16 + (P + 1) * 8, ms, peak, nnz=nnz[0],
                                               n_parts=P, buffer_sets=sets, l2_resident=resident,
                                               launches_per_call=LAUNCHES["partition"])
            launches += (steps + warmup) * sets * LAUNCHES["partition"]
            del p_out
        if wanted(sel, "next_c4_densify"):
            # group densification of the C4 lists (keys only)
            dn = [(torch.empty(zr.zr_densification_workspace_size(n, m), dtype=torch.uint8,
                               device=dev),
                   torch.empty(n.bit_length(), dtype=torch.int64, device=dev)) for _ in d_sets]
            stream = torch.cuda.current_stream().cuda_stream
            calls = [(lambda i, s=s, w=w: zr.zr_densification(
                [a.data_ptr() for a in s[0]], nnz, n, m, w[1].data_ptr(), w[0].data_ptr(),
                w[0].numel(), stream)) for s, w in zip(d_sets, dn)]
            ms = time_calls(torch, calls, steps, warmup)
            parts["next_c4_densify"] = part_entry(sum(nnz) * 4 + n.bit_length() * 8, ms, peak,
                                                  buffer_sets=sets, l2_resident=resident)
            launches += (steps + warmup) * sets * LAUNCHES["densify"]
            del dn
        if wanted(sel, "next_c4_hb"):
            # Zen's Pull: hash bitmaps of the union's keys over M = 2^25.  The
            # encode / decode go over all M indices through the directory's
            # slices (bound by that arithmetic: indices_per_s); their bytes are
            # the keys and the bitmaps.
            hb = zr.HashBitmap(m, P, seed)
            keys = d_sets[0][2].out_idx[:union]
            hb.encode(keys)
            hb_out = torch.empty(union, dtype=torch.int32, device=dev)
            hb_koff = torch.empty(P + 1, dtype=torch.int64, device=dev)
            hb_bits = hb.bits.clone()
            words = (m + 31) // 32
            dir_bytes = zr.zr_hash_directory_size(m, P)
            stream = torch.cuda.current_stream().cuda_stream
            ms = time_calls(torch, [lambda i: zr.zr_hash_directory(
                m, P, seed, hb.directory.data_ptr(), dir_bytes, stream)], steps, warmup)
            parts["next_c4_hb_directory"] = part_entry(dir_bytes, ms, peak,
                                                       indices_per_s=m / (ms / 1e3))
            ms = time_calls(torch, [lambda i: hb.encode(keys)], steps, warmup)
            parts["next_c4_hb_encode"] = part_entry(union * 4 + words * 4 + (P + 1) * 8, ms, peak,
                                                    indices_per_s=m / (ms / 1e3))
            ms = time_calls(torch, [lambda i: hb.decode(hb_bits, hb_out, hb_koff)], steps, warmup)
            parts["next_c4_hb_decode"] = part_entry(words * 4 + union * 4 + (P + 1) * 8, ms, peak,
                                                    indices_per_s=m / (ms / 1e3))
            sets = torch.empty(m, dtype=torch.int32, device=dev)
            offs = torch.empty(P + 1, dtype=torch.int64, device=dev)
            sets_ws = torch.empty(zr.zr_partition_workspace_size(m, P), dtype=torch.uint8,
                                  device=dev)
            ms = time_calls(torch, [lambda i: zr.zr_hash_index_sets(
                m, P, seed, sets.data_ptr(), offs.data_ptr(), sets_ws.data_ptr(),
                sets_ws.numel(), stream)], steps, warmup)
            parts["next_c4_hb_sets"] = part_entry(m * 4 + (P + 1) * 8, ms, peak)
            launches += (steps + warmup) * (LAUNCHES["hb_directory"] + LAUNCHES["hb_encode"]
                                            + LAUNCHES["hb_decode"] + LAUNCHES["hb_sets"])
            del hb, hb_out, hb_bits, sets, sets_ws
        del d_sets
        free()

    # ---- C5b: DGC top-5 % lists of 16 ranks (288 MB of input: no copies needed)
    if wanted(sel, "c5b") or wanted(sel, "next_c5b"):
        c = workloads.DGC_C5B
        m, P, seed = c["m"], c["n_parts"], c["part_seed"]
        idx_l, val_l = workloads.dgc_c5b()
        n = len(idx_l)
        nnz = [a.size for a in idx_l]
        di = [torch.from_numpy(a).to(dev) for a in idx_l]
        dv = [torch.from_numpy(v).to(dev) for v in val_l]
        work = zr.SparseWorkspace(n, m, P, sum(nnz), dev)
        zr.sparse_aggregate(di, dv, m, P, seed, work=work)
        torch.cuda.synchronize()
        union = int(work.out_nnz.item())
        if wanted(sel, "c5b_union"):
            ms = time_calls(torch, [lambda i: zr.sparse_aggregate(di, dv, m, P, seed, work=work)],
                            steps, warmup)
            parts["c5b_union"] = part_entry(sum(nnz) * 8 + union * 8 + (P + 1) * 8 + 8, ms, peak,
                                            n=n, m=m, union=union, n_parts=P,
                                            launches_per_call=LAUNCHES["union"])
            launches += (steps + warmup + 1) * LAUNCHES["union"]
        if wanted(sel, "next_c5b_densify"):
            w = torch.empty(zr.zr_densification_workspace_size(n, m), dtype=torch.uint8,
                            device=dev)
            o = torch.empty(n.bit_length(), dtype=torch.int64, device=dev)
            stream = torch.cuda.current_stream().cuda_stream
            ms = time_calls(torch, [lambda i: zr.zr_densification(
                [a.data_ptr() for a in di], nnz, n, m, o.data_ptr(), w.data_ptr(), w.numel(),
                stream)], steps, warmup)
            parts["next_c5b_densify"] = part_entry(sum(nnz) * 4 + n.bit_length() * 8, ms, peak)
            launches += (steps + warmup) * LAUNCHES["densify"]
        del di, dv, work
        free()

    # ---- C5a: the dense fp32 sweep N x M, ring all-reduce with the 1/N average
    if wanted(sel, "c5a"):
        for n in workloads.SWEEP_NS:
            for m in workloads.SWEEP_MS:
                name = "c5a_n%d_m2^%d" % (n, m.bit_length() - 1)
                if not wanted(sel, name):
                    continue
                set_bytes = n * m * 4
                sets, resident = rotation_sets(set_bytes)
                x = workloads.dense_device(n, m * sets, 1e-3, 500 + n, dev)
                # copy s is columns [s m, (s + 1) m) of every rank's row
                calls = [(lambda i, s=s: zr.ring_allreduce(
                    [x[r, s * m:(s + 1) * m] for r in range(n)], average=True))
                    for s in range(sets)]
                ms = time_calls(torch, calls, steps, warmup, graph=True)
                parts[name] = part_entry(
                    2 * n * m * 4, ms, peak, n=n, m=m, dtype="f32", buffer_sets=sets,
                    l2_resident=resident)
                launches += (steps + warmup + 1) * sets
                del x, calls
                free()
    return parts, launches


# ---------------------------------------------------------------- oracle
def oracle_sample(budget_s=12.0):
    """Time the CPU oracle, as it stands, on a bounded sample of the step's
    workload: the three Random SkipReduce calls (k = 0, 2, 4) of the C3
    configuration on the first M' bf16 elements of every rank (M' a multiple
    of N).  Returns a dict with the GB/s over the sample's algorithmic
    bytes."""
    import workloads
    from oracle import ring as oring

    c = workloads.DENSE_C3
    n = c["n"]
    mp = 1 << 20
    x = workloads.dense_bf16_per_rank(n, mp, c["sigma"], 300)
    nbytes = 0
    t_total = 0.0
    reps = 0
    t_start = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        y = x
        for k in C3_KS:
            o = oring.skip_offset(oring.SKIP_RANDOM, k, 0, reps, n)
            y = oring.allreduce_bf16(y, k=k, o=o, divisor=oring.DIV_N)
            nbytes += (n - k) * mp * 2 + n * mp * 2
        t_total += time.perf_counter() - t0
        reps += 1
        if time.perf_counter() - t_start > budget_s:
            break
    return {
        "value": nbytes / t_total / 1e9,
        "unit": UNIT,
        "cores": 1,
        "kind": "oracle",
        "sample": ("%d repetitions of the step's three Random SkipReduce calls (k = 0, 2, 4) on "
                   "8 ranks x %d bf16 (the first %d elements of each C3 rank); literal ring, "
                   "numpy, single-threaded" % (reps, mp, mp)),
        "seconds": t_total,
        "host_threads_available": len(os.sched_getaffinity(0)),
    }


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    res = oracle_sample(budget_s=max(5.0, min(60.0, 4.0 * args.steps)))
    line = {
        "impl": "reference", "metric": METRIC, "value": res["value"], "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": res["sample"]},
        "cpu_baseline": res,
        "e2e": {"value": res["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- main
def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch

    import __graft_entry__

    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    __graft_entry__.build()
    import gradient_synchronisation_gb300 as zr

    peak, peak_kind = measured_hbm()
    if args.parts_only:
        parts, n_launch = run_parts(torch, zr, dev, args.parts, max(1, args.steps),
                                    max(1, args.warmup), peak, None)
        if rank == 0:
            print(json.dumps({"profiling": args.parts, "steps": args.steps, "peak": peak,
                              "parts": parts, "gpu_launches": n_launch}))
        return 0
    S = Step(torch, zr, dev)
    step_bytes = S.bytes()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    total_ms, per = timed_step(torch, S, args.steps, args.warmup)
    if world > 1:
        total_ms = max_over_ranks(total_ms, dist, dev)
        dist.barrier()
    torch.cuda.synchronize()
    step_clk = clocks.stop()

    value = job_throughput(step_bytes, args.steps, world, total_ms)
    parts = {}
    for k in C3_KS:
        ms = statistics.median(per[k])
        parts["c3_k%d" % k] = part_entry(S.launch_bytes(k), ms, peak, n=S.n, m=S.m, dtype="bf16",
                                         k=k, skip_fraction=k / S.n)

    # Dominant kernel: ring_fused_kernel<bf16>, the k = 0 launch (the plain
    # ring with the average).  achieved = its algorithmic bytes over its
    # mean CUDA-event duration; the first timed launch also holds the host's
    # enqueue of the first step and is left out.
    k0 = per[0][1:] if len(per[0]) > 1 else per[0]
    ring_ms = statistics.mean(k0)
    achieved = S.launch_bytes(0) / (ring_ms / 1e3) / 1e9
    tr = TRAFFIC["ring_fused_kernel<bf16>"]
    sha = source_sha(os.path.join(ROOT, "gradient_synchronisation_gb300", "csrc", "ring.cu"))
    traffic = tr["bytes_per_launch"] if tr["source_sha256"] == sha else None

    e2e = None
    if not args.no_e2e:
        steps_e = max(2, min(args.steps, 5))
        e_ms, h2d, d2h = timed_e2e(torch, S, steps_e)
        e2e = {"value": world * step_bytes * steps_e / (e_ms / 1e3) / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    del S
    torch.cuda.empty_cache()
    part_launches = 0
    parts_clk = None
    if args.parts != "none":
        clocks = ClockSampler(torch.cuda.current_device())
        clocks.start()
        more, part_launches = run_parts(torch, zr, dev, args.parts, max(5, min(args.steps, 20)),
                                        max(3, args.warmup), peak, None)
        parts_clk = clocks.stop()
        parts.update(more)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_sample()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "bytes_per_step": step_bytes,
                       "l2": "inputs larger than L2 (8 rank buffers of 287 MB resident); the "
                             "parts smaller than twice the L2 are timed over copies of their "
                             "buffers used in turn (buffer_sets)",
                       "parallelism": "replicas only" if world > 1 else "single GPU",
                       "parts": "c3_* from the timed step; every other part timed after it, "
                                "in the same process, median of CUDA-event samples"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": "ring_fused_kernel<bf16>, C3 k = 0 launch",
                         "launches_averaged": len(k0), "peak_source": peak_kind},
            "parts": parts,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": step_clk,
            "clocks_parts": parts_clk,
            "gpu_launches": len(C3_KS) * args.steps,
            "gpu_launches_parts": part_launches,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
