#!/usr/bin/env python3
"""Benchmark of the batched generated-topology pass (one JSON line on stdout).

Workload (default): stress_b64_res512 -- B=64 members at resolution 512,
even members one-voxel-thick ellipsoid shells (semi-axes U[0.05,0.12]*512),
odd members Bernoulli(0.02) blobs in boxes of side U{64..128}, every member
moved to straddle a +-4096 root-tile boundary in one of the eight sign
octants (1.31 M input voxels).  It is the largest of the workloads, all of
which fit one GPU; the B=16 and B=48 shell batches of fVDB PR #757's
"Measurements" (~7.8k voxels per member, resolution 64, median of 20
CUDA-event iterations) are timed per call in the ``per_op`` table and the
``target`` block.

One step runs every pass of the hot path once over the batch, each through
the library's C ABI:
  from_ijk (ijk front end), refine x2 (conv_transpose_grid k2s2),
  coarsen x2 (conv_grid k2s2), dilate [-1,1]^3 (conv_grid k3s1), the two pad
  octants {-1,0}^3 and {0,1}^3, the k3s2 transpose chain (refine x2 then the
  {-1,0}^3 pad) and coarsen x4 -- the front end, then one tb_multi call of the
  seven chains.
value = output voxels of the step's calls / device time of the step.

Legs: device-resident inputs (value); end to end from pinned host memory with
the results read back (e2e); a repetition with per-kernel CUDA events for the
roofline of the dominant kernel (algorithmic bytes per pass: 76 per source
leaf, 116 per output leaf, 24 per slot per digit pass); the CPU oracle on a
bounded sample (cpu_baseline: one thread, primary; all host threads,
secondary).  ``--impl reference`` times the oracle alone (the reference arm
of this benchmark).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "output voxels/s per batched topology pass (device-timed); % of HBM roofline"
UNIT = "voxels/s"
DIL = ("dilate", (-1, -1, -1), (1, 1, 1))
PAD_N = ("dilate", (-1, -1, -1), (0, 0, 0))
PAD_P = ("dilate", (0, 0, 0), (1, 1, 1))
# (label, ops of the call); an empty op list is the from_ijk front end
STEP = [("from_ijk", []), ("refine2", [("refine", 2)]), ("coarsen2", [("coarsen", 2)]),
        ("dilate_k3s1", [DIL]), ("pad_neg", [PAD_N]), ("pad_pos", [PAD_P]),
        ("k3s2", [("refine", 2), PAD_N]), ("coarsen4", [("coarsen", 4)])]
L2_FLUSH_BYTES = 256 << 20


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="stress_b64_res512")
    p.add_argument("--no-extra", action="store_true", help="skip the per-op and larger-workload tables")
    p.add_argument("--cpu-sample-members", type=int, default=16,
                   help="members of the batch in the single-thread oracle sample (0: no CPU baseline)")
    p.add_argument("--separate", action="store_true", help="one C-ABI call per chain instead of one tb_multi call")
    p.add_argument("--phases", action="store_true",
                   help="only the step's per-call phase breakdown (GPU timer stamps and host timers)")
    p.add_argument("--kmap-only", action="store_true",
                   help="only the kernel-map rows, in every kernel form, on the B=16 and B=48 shells and the "
                        "stress batch")
    p.add_argument("--kmap-workloads", default="shells_b16_res64,shells_b48_res64,stress_b64_res512",
                   help="--kmap-only: comma-separated workloads")
    p.add_argument("--kmap-forms", default="auto,staged,staged_prepass,tabulated,per_entry",
                   help="--kmap-only: comma-separated kernel forms (tb.set_kmap_mode)")
    return p.parse_args()


# ------------------------------------------------------------------ helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class Clocks:
    """Samples nvidia-smi every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", "tb_clocks_%d_%d.csv" % (os.getpid(), index))

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except Exception:
            return None
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def kernel_traffic(name):
    """DRAM bytes per launch of `name` from the committed ncu summary, if the
    kernel sources are unchanged since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))
    except Exception:
        return None
    if d.get("source_hash") != source_hash():
        return None
    k = d.get("kernels", {}).get(name)
    return None if k is None else k.get("dram_bytes_per_launch")


def source_hash():
    """Hash of the sources of the pass kernels and the calls that plan them
    (every CUDA source but the kernel maps'): traffic figures taken before a
    change there no longer describe the kernel."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_voxel_grid_leaf_gb300", "csrc")
    for n in sorted(os.listdir(csrc)):
        if n.endswith((".cu", ".cuh", ".h")) and n != "tb_kmap.cu":
            h.update(open(os.path.join(csrc, n), "rb").read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ CPU oracle

def oracle_step(ijk, off, threads, members=None):
    """One step of the oracle over the given members (default: all), the
    members spread over `threads` threads (members are independent; the
    oracle itself is unchanged).  Returns the output voxels of the step's
    calls on those members (the metric's count)."""
    import concurrent.futures as cf
    import numpy as np
    import oracle
    B = len(off) - 1
    members = range(B) if members is None else members
    subs = [(ijk[off[g]:off[g + 1]], np.array([0, off[g + 1] - off[g]], np.int64)) for g in members]

    def one(args):
        sub, o, ops = args
        return int(oracle.run_voxels(sub, o, ops)["voxel_counts"].sum())

    jobs = [(sub, o, ops) for _, ops in STEP for sub, o in subs]
    if threads == 1:
        return sum(map(one, jobs))
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        return sum(ex.map(one, jobs))


def host_cores():
    """(nproc: threads this process may run on, hardware threads of the host
    -- std::thread::hardware_concurrency)."""
    return cpu_threads(), os.cpu_count() or 1


def cpu_baseline(ijk, off, n_members):
    """The oracle, as it stands, on a bounded sample of the workload: the
    step's eight calls on members 0..n_members-1 with one thread (primary:
    the oracle is single-threaded), and on all members spread over every
    host thread (secondary).  voxels/s is the metric's unit."""
    B = len(off) - 1
    sample = list(range(min(n_members, B)))
    nproc, hw = host_cores()
    t0 = time.perf_counter()
    v1 = oracle_step(ijk, off, 1, sample)
    dt1 = time.perf_counter() - t0
    t0 = time.perf_counter()
    vn = oracle_step(ijk, off, nproc)
    dtn = time.perf_counter() - t0
    return {"value": v1 / dt1, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "one step (all eight calls) on members 0-%d of %d, one thread: %d output voxels in %.1f s"
                      % (len(sample) - 1, B, v1, dt1),
            "nproc": nproc, "hardware_concurrency": hw,
            "threaded": {"value": vn / dtn, "unit": UNIT, "cores": nproc,
                         "sample": "one full step (all %d members), members over %d threads: %.1f s"
                                   % (B, nproc, dtn)}}


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ reference arm

REF_MEMBERS_PER_STEP = 16


def run_reference(args):
    """The oracle timed alone on this arm's workload and metric: each step is
    the eight calls on a block of REF_MEMBERS_PER_STEP members (rotating
    through the batch from step to step), members over every host thread."""
    from sparse_voxel_grid_leaf_gb300 import synth
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    ijk, off = synth.make(args.workload)
    B = len(off) - 1
    threads, hw = host_cores()
    per = min(REF_MEMBERS_PER_STEP, B) if B else 0

    def block(i):
        return [(i * per + j) % B for j in range(per)] if B else []
    for i in range(args.warmup):
        oracle_step(ijk, off, threads, block(i))
    t0 = time.perf_counter()
    vox = 0
    for i in range(args.steps):
        vox += oracle_step(ijk, off, threads, block(args.warmup + i))
    dt = time.perf_counter() - t0
    value = vox / dt
    sample = ("each step: the eight calls on %d of the %d members (a rotating block), members over %d threads"
              % (per, B, threads))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
            "data": "synthetic", "config": {"workload": args.workload, "step": [s for s, _ in STEP],
                                            "members_per_step": per},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
                             "nproc": threads, "hardware_concurrency": hw},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

SEPARATE = False  # --separate: one C-ABI call per chain instead of one tb_multi call


def run_step(tb, b_src, inputs):
    """Runs the step: the ijk front end, then every chain on its output (one
    tb_multi call, or one call per chain); returns the batches by label."""
    out = {}
    b0 = tb.from_ijk(*inputs)
    out["from_ijk"] = b0
    if SEPARATE:
        for label, ops in STEP[1:]:
            out[label] = tb.chain(b0, ops)
    else:
        global _PLAN
        if _PLAN is None:
            _PLAN = tb.MultiPlan([ops for _, ops in STEP[1:]])
        for (label, _), b in zip(STEP[1:], _PLAN(b0)):
            out[label] = b
    return out


_PLAN = None  # the step's chains, marshalled once


def step_voxels(outs):
    """Output voxels of the step: the outputs of its eight calls (a chain counts
    its result only; its passes are fused, so no intermediate is produced)."""
    v = {k: int(b.to_numpy(["voxel_counts"])["voxel_counts"].sum()) for k, b in outs.items()}
    return sum(v.values()), v


def free_all(outs):
    for b in outs.values():
        b.free()


def pass_stats(outs):
    """Per pass (L_in, S, L_out, P, NL, NU, kind) for the byte model.  Every
    call of the step is one pass but k3s2 (refine x2 then the {-1,0}^3 pad):
    the library fuses it into one pass for inputs of at most 32,768 leaves,
    and runs its two passes otherwise (a batch built by more than one pass
    reports -1 source leaves).  Its first pass then equals the refine x2
    call of the same step (same input, same op), so that call's counts stand
    for it; coarsen x4 is always one pass."""
    b0 = outs["from_ijk"]
    ps = []

    def add(kind, L_in, b, S=None, L_out=None):
        ps.append({"kind": kind, "L_in": L_in, "S": b.build_slots if S is None else S,
                   "L_out": b.num_leaves if L_out is None else L_out,
                   "P": model_digit_passes(b), "P_run": b.build_digit_passes, "NL": b.num_lowers,
                   "NU": b.num_uppers, "B": b.num_grids, "kernel": "member" if b.build_member_ctas else "chain"})
    add("ijk", b0.build_source_leaves, b0)
    add("refine", b0.num_leaves, outs["refine2"])
    add("coarsen", b0.num_leaves, outs["coarsen2"])
    add("dilate", b0.num_leaves, outs["dilate_k3s1"])
    add("dilate", b0.num_leaves, outs["pad_neg"])
    add("dilate", b0.num_leaves, outs["pad_pos"])
    k3 = outs["k3s2"]
    if k3.build_source_leaves < 0:
        r2 = outs["refine2"]
        # its refine pass, handing its leaves to the pad pass (no writer)
        ps.append(dict(ps[1], kernel="member" if k3.build_member_ctas else "chain", inter=True))
        add("dilate", r2.num_leaves, k3)
    else:
        add("refine_dilate", b0.num_leaves, k3)
    add("coarsen", b0.num_leaves, outs["coarsen4"])
    return ps


def kernel_bytes(ps):
    """Algorithmic DRAM bytes per kernel over one step (each record read or
    written once; per-grid arrays ignored).  "chain" is the cooperative
    whole-grid pass kernel of a call and "member" the member launch (one
    cluster per grid), whichever built the pass: emission, digit passes,
    index, leaves and voxel offsets of each of its passes; "write_<op>" is the
    final writer of a one-chain call, "write_multi" the one writer of all
    chains of a tb_multi call.

    Per pass, with L_in source leaves (voxels for the ijk front end), S slots,
    L_out unique leaves and P digit passes:
      front end  the input's bbox: 12 B per voxel (ijk front end)
      emission   source records (80 B: origin, mask, grid; 12 B per voxel) + 12 S
      sort       24 S P (key and reference read and written per digit pass)
      index      8 S (keys) + 12 L_out (run start, lower and upper index)
      leaves     20 L_out + 4 S + the source masks again (64 B per source
                 leaf; an ijk slot carries its voxel's bit), then 80 L_out
                 hand-off (intermediate) or 84 L_out staged record, popcount
                 and grid (last)
      writer     96 L_out read (staged record, grid, voxel offset, node
                 indices) + 124 L_out written + 16 per lower + 12 per upper
    """
    by = {}

    def acc(name, n):
        by[name] = by.get(name, 0) + n
    for p in ps:
        L_in, S, L_out = p["L_in"], p["S"], p["L_out"]
        ijk = p["kind"] == "ijk"
        src = 24 * L_in if ijk else 80 * L_in     # ijk: the bbox read, then the emission's
        merge = 20 * L_out + 4 * S + (0 if ijk else 64 * L_in)
        chain = src + 12 * S + 24 * S * p["P"] + 8 * S + 12 * L_out + merge
        chain += 80 * L_out if p.get("inter") else 84 * L_out
        acc(p.get("kernel", "chain"), chain)
        if not p.get("inter"):
            w = "write_" + p["kind"] if SEPARATE or ijk else "write_multi"
            acc(w, 96 * L_out + 124 * L_out + 16 * p["NL"] + 12 * p["NU"])
    return by


def model_digit_passes(b):
    """P of the byte model: the 8-bit digit passes a radix sort over the key
    bits that vary across the batch takes, ceil(W / 8) for the pass's
    compressed key of W bits -- a property of the workload, whichever way the
    library orders the leaves (the lower-node child-mask path runs none)."""
    return (b.build_key_bits + 7) // 8


def pass_bytes(p):
    """Algorithmic bytes of one pass: each source record read once (76 B per
    source leaf: origin and 64-byte mask; 12 B per voxel for the ijk front
    end), each output leaf record written once (116 B: origin, mask, voxel
    offset, word prefix, leaf bbox), each slot's 8-byte key and 4-byte source
    reference read and written once per digit pass (24 B per slot per pass),
    and about 100 B of per-grid arrays per grid."""
    src = 12 * p["L_in"] if p["kind"] == "ijk" else 76 * p["L_in"]
    return src + 116 * p["L_out"] + 24 * p["S"] * p["P"] + 100 * p["B"]


def pass_model_bytes(ps):
    """Whole-step byte model: the sum of pass_bytes over the step's passes."""
    return sum(pass_bytes(p) for p in ps)


def rank_batch(synth, workload, rank):
    """Weak scaling: every rank builds its own batch of the workload's shape
    (same generator parameters, seed = rank)."""
    return synth.make(workload, seed=rank)


def job_totals(dist, total_ms, voxels, device):
    """(slowest rank's timed milliseconds, output voxels of all ranks): the
    ranks process independent batches, so the job's throughput is the sum of
    their work over the longest of their times."""
    if dist is None:
        return float(total_ms), float(voxels)
    import torch
    t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    v = torch.tensor([float(voxels)], dtype=torch.float64, device=device)
    dist.all_reduce(v)
    return float(t.item()), float(v.item())


def run_ours(args):
    import numpy as np
    import torch
    import sparse_voxel_grid_leaf_gb300 as tb
    from sparse_voxel_grid_leaf_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    tb.lib()
    stream = torch.cuda.current_stream()
    if args.kmap_only:
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        if rank == 0:
            print(json.dumps({"per_op": kmap_table(tb, torch, synth, stream, flush,
                                                   args.kmap_workloads.split(","), args.kmap_forms.split(","))}),
                  flush=True)
        return
    if args.phases:
        if rank == 0:
            print(json.dumps({"phases": phase_table(tb, torch, synth, args.workload, args.steps)}), flush=True)
        return

    ijk, off = rank_batch(synth, args.workload, rank)
    ijk_d = torch.from_numpy(ijk).cuda()
    off_d = torch.from_numpy(off).cuda()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    # ---- warm-up and the step's output size
    for _ in range(max(args.warmup, 3)):
        outs = run_step(tb, None, (ijk_d, off_d))
        free_all(outs)
    outs = run_step(tb, None, (ijk_d, off_d))
    voxels, per_label = step_voxels(outs)
    ps = pass_stats(outs)
    out_leaves = {k: (b.num_grids, b.num_leaves) for k, b in outs.items()}
    free_all(outs)
    torch.cuda.synchronize()

    # ---- timed region: device-resident inputs
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = tb.kernel_launch_count()
    times = []
    with Clocks(local) as clk:
        for _ in range(args.steps):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            outs = run_step(tb, None, (ijk_d, off_d))
            e.record(stream)  # the step ends with its outputs written; freeing them is the caller's later business
            e.synchronize()
            free_all(outs)
            times.append(s.elapsed_time(e))
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    launches = tb.kernel_launch_count() - launches0
    total_ms, job_voxels = job_totals(dist, sum(times), voxels, "cuda")
    value = job_voxels * args.steps / (total_ms / 1e3)
    ms_per_step = total_ms / args.steps

    # ---- end to end: pinned host inputs in, leaf records back to pinned host memory
    ijk_h = torch.from_numpy(ijk).pin_memory()
    off_h = torch.from_numpy(off).pin_memory()
    host_out = {k: (torch.empty((L, 3), dtype=torch.int32).pin_memory(),
                    torch.empty((L, 8), dtype=torch.int64).pin_memory(),
                    torch.empty((L,), dtype=torch.int64).pin_memory(),
                    torch.empty((B + 1,), dtype=torch.int64).pin_memory()) for k, (B, L) in out_leaves.items()}
    d2h = sum(12 * L + 64 * L + 8 * L + 8 * (B + 1) for B, L in out_leaves.values())
    h2d = ijk_h.numel() * 4 + off_h.numel() * 8
    keys = [k for k, _ in STEP]
    export = tb.ExportPlan([host_out[k][0] for k in keys], [host_out[k][1] for k in keys],
                           [host_out[k][2] for k in keys], [host_out[k][3] for k in keys])
    # The steps run as an application's loop would: step i's export, on a
    # copy stream, overlaps step i+1's compute (arrays of 1 MiB or more go
    # through the copy engines, so the export takes no SM time).  A step's
    # outputs are freed once its export is done, after the next step has
    # been enqueued.  No L2 flush: the inputs come from host memory and a
    # step's device working set (107 MB of outputs alone at stress size)
    # exceeds the L2.  Timed from before the first step's first call to the
    # end of the last export, on the device.
    copy = torch.cuda.Stream()

    def e2e_steps(n):
        pending = None
        for _ in range(n):
            outs = run_step(tb, None, (ijk_h, off_h))
            ready = torch.cuda.Event()
            ready.record(stream)
            copy.wait_event(ready)
            export([outs[k] for k in keys], stream=copy)
            exported = torch.cuda.Event()
            exported.record(copy)
            if pending is not None:
                stream.wait_event(pending[1])
                free_all(pending[0])
            pending = (outs, exported)
        return pending

    last = e2e_steps(args.warmup)
    if last is not None:
        stream.wait_event(last[1])
        free_all(last[0])
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    last = e2e_steps(args.steps)
    e.record(copy)
    e.synchronize()
    if last is not None:
        stream.wait_event(last[1])
        free_all(last[0])
    torch.cuda.synchronize()
    e2e_times = [s.elapsed_time(e) / args.steps] * args.steps
    e2e_ms, _ = job_totals(dist, sum(e2e_times), voxels, "cuda")
    e2e_value = job_voxels * len(e2e_times) / (e2e_ms / 1e3)

    # ---- roofline of the dominant kernel (instrumented repetition)
    peak, peak_kind = measured_peaks()
    reps = max(3, min(args.steps, 10))
    tb.profile_read()
    tb.profile_enable(True)
    for _ in range(reps):
        flush.zero_()
        outs = run_step(tb, None, (ijk_d, off_d))
        free_all(outs)
    torch.cuda.synchronize()
    prof = tb.profile_read()
    tb.profile_enable(False)
    kb = kernel_bytes(ps)
    tot_kernel_ms = sum(ms for _, ms in prof.values())
    dom = max(prof, key=lambda k: prof[k][1])
    n_launch, dom_ms = prof[dom]
    # algorithmic bytes of the passes the dominant (pass) kernel runs per step
    dom_passes = [p for p in ps if p.get("kernel") == dom]
    bytes_step = sum(pass_bytes(p) for p in dom_passes)
    achieved = bytes_step * reps / (dom_ms / 1e3) / 1e9
    traffic = kernel_traffic(dom)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "kernel": dom,
                "bytes_per_launch": bytes_step * reps / n_launch, "us_per_launch": 1e3 * dom_ms / n_launch,
                "launches_per_step": n_launch / reps,
                "bytes_model": "per pass 76 L_in + 116 L_out + 24 S P + 100 B (12 per voxel for an ijk source)",
                "passes": [{k: p[k] for k in ("kind", "L_in", "S", "P", "P_run", "L_out", "B")} for p in dom_passes],
                "share_of_kernel_time": dom_ms / tot_kernel_ms, "peak_source": peak_kind + " hbm_gbs (copy)"}
    kernels = {k: {"launches_per_step": n / reps, "us_per_launch": 1e3 * ms / n,
                   "share": ms / tot_kernel_ms,
                   "phase_model_GBps": (kb.get(k, 0) * reps / (ms / 1e3) / 1e9) if kb.get(k) else None}
               for k, (n, ms) in sorted(prof.items(), key=lambda kv: -kv[1][1])}
    model = pass_model_bytes(ps)

    # ---- CPU oracle on a bounded sample (rank 0, one GPU only)
    cpu = None
    if rank == 0 and world == 1 and args.cpu_sample_members > 0:
        cpu = cpu_baseline(ijk, off, args.cpu_sample_members)

    # ---- per-op and larger-workload tables (median of 20 after 5 warm-ups)
    extra = {}
    if not args.no_extra and rank == 0:
        extra = per_op_tables(tb, torch, synth, stream, flush, args.workload)

    if rank != 0:
        return
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "config": {"workload": args.workload, "B": len(off) - 1, "input_voxels": int(len(ijk)),
                       "step": [s for s, _ in STEP], "passes_per_step": len(ps),
                       "output_voxels_per_step": voxels, "output_voxels_by_call": per_label,
                       "l2": "flushed before every step (256 MB write, untimed)", "inputs": "device-resident",
                       "calls": "from_ijk + one call per chain" if SEPARATE else "from_ijk + one tb_multi call"},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms / len(e2e_times),
                    "mode": "pipelined: step i's export to pinned host memory on a copy stream overlaps step "
                            "i+1; inputs read from pinned host memory by the front end; no L2 flush"},
            "roofline": roofline,
            "pass_model": {"bytes_per_step": model, "GBps": model / (ms_per_step / 1e3) / 1e9,
                           "frac": model / (ms_per_step / 1e3) / 1e9 / peak},
            "kernels": kernels, "gpu_launches": launches, "cpu_baseline": cpu,
            "clocks": clk.summary(), "target": target_block(extra, peak), "per_op": extra}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def per_op_tables(tb, torch, synth, stream, flush, main_workload):
    """ms per call (median of 20 CUDA-event iterations after 5 warm-ups, L2
    flushed before each) for each single call on three workloads: the pages'
    conv-grid ops, the fused chains, masked refinement (half the voxels
    flagged), a K=5 stride-1 topology, and two kernel maps (with the GB/s of
    the map they write)."""
    import numpy as np
    res = {}
    ops = [("refine2", [("refine", 2)]), ("coarsen2", [("coarsen", 2)]), ("dilate_k3s1", [DIL]),
           ("pad_neg", [PAD_N]), ("k3s2", [("refine", 2), PAD_N]), ("coarsen4", [("coarsen", 4)]),
           ("conv_k5s1", [("dilate", (-2, -2, -2), (2, 2, 2))])]
    for wl in dict.fromkeys(("shells_b16_res64", "shells_b48_res64", "stress_b64_res512", main_workload)):
        ijk, off = synth.make(wl)
        ijk_d, off_d = torch.from_numpy(ijk).cuda(), torch.from_numpy(off).cuda()
        b0 = tb.from_ijk(ijk_d, off_d)
        fine = tb.refine(b0)
        V = int(b0.to_numpy(["voxel_counts"])["voxel_counts"].sum())
        flags = torch.from_numpy((np.random.default_rng(0).random(V) < 0.5).astype(np.uint8)).cuda()
        plan = tb.MultiPlan([o for _, o in ops[:5]])
        row = {}
        calls = [("from_ijk", lambda: tb.from_ijk(ijk_d, off_d))] + \
                [(lab, (lambda o=o: tb.chain(b0, o))) for lab, o in ops] + \
                [("multi5", lambda: plan(b0)),
                 ("refine_masked_half", lambda: tb.refine_masked(b0, flags)),
                 ("kmap_k3s1", lambda: tb.kernel_map(b0, b0)),
                 ("kmap_k2s2_transpose", lambda: tb.kernel_map(b0, fine, (0, 0, 0), (1, 1, 1), 2, True))]
        row = time_calls(calls, torch, stream, flush)
        res[wl] = row
        fine.free()
        b0.free()
    res["pyramid_b48_res64"] = pyramid_table(tb, torch, synth, stream, flush)
    return res


def time_calls(calls, torch, stream, flush):
    """{label: row} for (label, fn) calls: median ms of 20 CUDA-event
    iterations after 5 warm-ups, L2 flushed before each; a call returning a
    tensor (a kernel map) reports the GB/s of the map it writes, one returning
    batches their output voxels per second."""
    row = {}
    for lab, fn in calls:
        ts = []
        vox = 0
        nbytes = 0
        stats = None
        for it in range(25):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            r = fn()
            e.record(stream)
            e.synchronize()
            if isinstance(r, torch.Tensor):
                nbytes = r.numel() * 4
                del r
            else:
                rs = r if isinstance(r, list) else [r]
                if it == 0:
                    vox = sum(int(x.to_numpy(["voxel_counts"])["voxel_counts"].sum()) for x in rs)
                    one = rs[0] if len(rs) == 1 else None
                    stats = None if one is None else {
                        "L_in": one.build_source_leaves, "S": one.build_slots, "P": model_digit_passes(one),
                        "P_run": one.build_digit_passes, "L_out": one.num_leaves, "B": one.num_grids}
                for x in rs:
                    x.free()
            if it >= 5:
                ts.append(s.elapsed_time(e))
        med = statistics.median(ts)
        if nbytes:
            row[lab] = {"ms": med, "map_bytes": nbytes, "map_GBps": nbytes / med / 1e6}
        else:
            row[lab] = {"ms": med, "out_voxels": vox, "Gvox_per_s": vox / med / 1e6}
            if stats is not None:
                row[lab]["last_pass"] = stats
    return row


def target_block(per_op, peak):
    """The single conv-grid calls at B=48 and at stress size against the HBM
    roofline: ms per call (median of 20, L2 flushed) and the call's
    algorithmic bytes (pass_bytes) over that time, as a fraction of the
    measured copy bandwidth.  Each of these calls is one pass."""
    out = {}
    kinds = {"refine2": "refine", "coarsen2": "coarsen", "dilate_k3s1": "dilate"}
    for wl in ("shells_b48_res64", "stress_b64_res512"):
        for lab, kind in kinds.items():
            r = (per_op.get(wl) or {}).get(lab)
            if not r or "last_pass" not in r:
                continue
            p = dict(r["last_pass"], kind=kind)
            nbytes = pass_bytes(p)
            gbps = nbytes / (r["ms"] / 1e3) / 1e9
            out["%s/%s" % (wl, lab)] = {"ms": r["ms"], "bytes": nbytes, "GBps": gbps, "frac": gbps / peak,
                                        "S": p["S"], "P": p["P"], "P_run": p.get("P_run"), "L_in": p["L_in"],
                                        "L_out": p["L_out"]}
    return out


def phase_table(tb, torch, synth, workload, steps):
    """Where a step's time goes, per call (the front end; the tb_multi call;
    refine x2, coarsen x2 and dilate [-1,1]^3 alone):
    mean microseconds per call of each kernel and of each pass-kernel phase
    (GPU global-timer stamps: entry to the first emission, emission, digit
    passes, index, leaves, voxel offsets) and of the host's share of the
    call, over `steps` steps after 5 warm-ups, without an L2 flush.  The
    stamps add a little to the kernels they time."""
    ijk, off = synth.make(workload)
    ijk_d, off_d = torch.from_numpy(ijk).cuda(), torch.from_numpy(off).cuda()
    plan = tb.MultiPlan([ops for _, ops in STEP[1:]])
    res = {}
    b0 = tb.from_ijk(ijk_d, off_d)
    calls = [("from_ijk", lambda: tb.from_ijk(ijk_d, off_d)), ("multi7", lambda: plan(b0))] + \
            [(lab, (lambda o=o: tb.chain(b0, o))) for lab, o in STEP[1:4]]
    for label, fn in calls:
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        tb.profile_read()
        tb.profile_enable(2)
        for _ in range(steps):
            fn()
        torch.cuda.synchronize()
        prof = tb.profile_read()
        tb.profile_enable(0)
        res[label] = {k: 1e3 * ms / steps for k, (n, ms) in prof.items()}
    return res


def kmap_table(tb, torch, synth, stream, flush, workloads, forms):
    """The kernel-map rows alone (as in per_op_tables) on the given
    workloads: the k3s1 same-topology map, then the k2s2 transpose map to
    the refinement, 25 calls each, in each given kernel form
    (tb.set_kmap_mode; "auto" is the form the library picks)."""
    res = {}
    for wl in workloads:
        ijk, off = synth.make(wl)
        b0 = tb.from_ijk(torch.from_numpy(ijk).cuda(), torch.from_numpy(off).cuda())
        fine = tb.refine(b0)
        res[wl] = {}
        for form in forms:
            prev = tb.set_kmap_mode(form)
            try:
                res[wl][form] = time_calls([("kmap_k3s1", lambda: tb.kernel_map(b0, b0)),
                                            ("kmap_k2s2_transpose",
                                             lambda: tb.kernel_map(b0, fine, (0, 0, 0), (1, 1, 1), 2, True))],
                                           torch, stream, flush)
            finally:
                tb.set_kmap_mode(prev)
        fine.free()
        b0.free()
    return res


PYRAMID = [("e1", [("coarsen", 2)]), ("e2", [("coarsen", 4)]), ("e3", [("coarsen", 8)]),
           ("u2", [("coarsen", 8), ("refine", 2)]),
           ("d2", [("coarsen", 8), ("refine", 2), DIL]),
           ("u1", [("coarsen", 8), ("refine", 2), DIL, ("refine", 2)]),
           ("d1", [("coarsen", 8), ("refine", 2), DIL, ("refine", 2), DIL]),
           ("u0", [("coarsen", 8), ("refine", 2), DIL, ("refine", 2), DIL, ("refine", 2)])]


def pyramid_table(tb, torch, synth, stream, flush):
    """The 4-level pyramid rebuild on pyramid_b48_res64 (encoder coarsenings
    by 2, 4, 8; decoder refinements with a k3s1 dilation per level; 11 passes
    of the pages' schedule): as 8 calls level by level, and as one tb_multi
    call of the 8 chains (one launch; fused passes).  Median ms of 20 after
    5 warm-ups, L2 flushed; the front end is not included."""
    ijk, off = synth.make("pyramid_b48_res64")
    b0 = tb.from_ijk(torch.from_numpy(ijk).cuda(), torch.from_numpy(off).cuda())
    plan = tb.MultiPlan([o for _, o in PYRAMID])

    def levels():
        e1, e2, e3 = tb.coarsen(b0, 2), tb.coarsen(b0, 4), tb.coarsen(b0, 8)
        u2 = tb.refine(e3)
        d2 = tb.box_dilate(u2)
        u1 = tb.refine(d2)
        d1 = tb.box_dilate(u1)
        u0 = tb.refine(d1)
        return [e1, e2, e3, u2, d2, u1, d1, u0]
    row = {}
    for lab, fn in (("pyramid_8_calls", levels), ("pyramid_one_multi", lambda: plan(b0))):
        ts = []
        vox = 0
        for it in range(25):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            rs = fn()
            e.record(stream)
            e.synchronize()
            if it == 0:
                vox = sum(int(x.to_numpy(["voxel_counts"])["voxel_counts"].sum()) for x in rs)
            for x in rs:
                x.free()
            if it >= 5:
                ts.append(s.elapsed_time(e))
        med = statistics.median(ts)
        row[lab] = {"ms": med, "out_voxels": vox, "Gvox_per_s": vox / med / 1e6}
    b0.free()
    return row


def main():
    global SEPARATE
    args = parse()
    SEPARATE = args.separate
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
