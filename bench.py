#!/usr/bin/env python
"""Benchmark of the MSA hot path on GB300; prints ONE JSON line (rank 0).

A step is one pass of the whole hot path over one batch of synthetic input:
  prefill at N = 131072 tokens (index block scores -> per-group top-k selection -> sparse main
  branch; H_q=32, H_kv=4, d_h=128, d_idx=64, block 64, k=16, 8 hot blocks), then
  decode of 32 sequences with cache lengths ~ U[65536, 262144] (same head layout).
`value` is prefill tokens/s (N / prefill device time); decode tokens/s is reported beside it, and
the forward of the KL alignment loss (on the step's selection and LSE), the decode of the same
batch from a paged KV cache, and a varlen prefill of the same tokens cut into sequences of mixed
lengths are timed after the steps, outside `value`.
Inputs stay resident in HBM; every timed input (M alone is 4.3 GB, the decode caches 11.5 GB)
is larger than the 129 MB L2, so no flush is needed.

--impl reference times the CPU oracle (the plain fp64 restatement of the formulas) on bounded
samples of the same prefill workload, on this host's cores.
Multi-process (torchrun): every rank runs its own replica of the workload on its own GPU
(weak scaling, no collective on the data path); times are max-reduced.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gen  # noqa: E402

METRIC = ("MSA prefill tokens/s and decode tokens/s at 128K ctx; % of bf16 TC / HBM roofline")
# kernels per step: the fused index branch (block scores + top-k); attention per 65536-row chunk:
# plan, scan, scatter, block-major pass, shared-block pass with the merge (+ one memset); decode:
# the index-key scan and the tail (selection + attention + merge in one kernel)
ATTN_LAUNCHES_PER_CHUNK = 5
ATTN_CHUNK_ROWS = 65536
DECODE_LAUNCHES = 2
KERNEL_FILES = {"index_branch": ["k_score.cu"],
                "main_branch": ["attn_fwd.cu", "k_attn_shared.cu", "k_attn_kvouter.cu",
                                "k_attn_plan.cu", "attn_tile.cuh"],
                "decode": ["k_decode.cu", "select_core.cuh", "k_attn.cu"],
                "kl_loss_fwd": ["k_kl.cu", "k_attn_plan.cu", "attn_tile.cuh"],
                "kl_loss_bwd": ["k_kl.cu", "k_attn_plan.cu", "attn_tile.cuh"],
                "sparse_attn_bwd": ["k_attn_bwd.cu", "k_kl.cu", "k_attn_plan.cu", "attn_tile.cuh"]}
# the KL alignment loss forward, timed apart from the step: plan, scan, plan, block-major pass,
# merge (+ two memsets); its gradient: row-ordered bucketing (count, scan, bases, scatter),
# block-major pass, dQ_idx merge, dK_idx merge (+ two memsets)
KL_LAUNCHES = 5
KLB_LAUNCHES = 7


# ------------------------------------------------------------------------ helpers --

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"],
                    bf16_sust=p.get("bf16_tflops_sustained", p["bf16_tflops"]), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


def kernel_source_hash(fnames):
    h = hashlib.sha256()
    for f in fnames:
        h.update(open(os.path.join(ROOT, "block_sparse_gqa_scores_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


# ncu kernel name -> the bench row it belongs to (a row is one call of the C ABI per step)
NCU_ROWS = {"k_index_block_scores": "index_branch",
            "k_attn_plan": "main_branch", "k_attn_scan": "main_branch",
            "k_attn_scatter": "main_branch",
            "k_attn_kvouter": "main_branch", "k_attn_shared": "main_branch",
            "k_decode_block_scores": "decode", "k_decode_tail": "decode",
            "k_kl_plan": "kl_loss_fwd", "k_kl_kvouter": "kl_loss_fwd", "k_kl_merge": "kl_loss_fwd",
            "k_kl_dq_merge": "kl_loss_bwd", "k_kl_dk_merge": "kl_loss_bwd",
            "k_attn_bwd_kvouter": "sparse_attn_bwd", "k_attn_bwd_dq_merge": "sparse_attn_bwd",
            "k_attn_bwd_dkv_merge": "sparse_attn_bwd", "k_attn_bwd_delta": "sparse_attn_bwd"}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")


DEFAULT_WORKLOAD = True   # cleared by run_msa for any other prefill/decode workload


def ncu_traffic(kernel):
    """DRAM bytes per call of a bench row from the last full-size ncu capture, if the row's
    kernel sources are unchanged since (profiles/traffic.txt records the source hash) and the
    bench runs the workload that capture was taken on."""
    if not DEFAULT_WORKLOAD or not os.path.exists(TRAFFIC_FILE):
        return None
    for line in open(TRAFFIC_FILE):
        f = line.split()
        if len(f) >= 3 and not line.startswith("#") and f[0] == kernel:
            return int(float(f[1])) if f[2] == kernel_source_hash(KERNEL_FILES[kernel]) else None
    return None


def write_traffic(csv_path, command, scale=1.0, only=None, tag="A"):
    """Updates profiles/traffic.txt from an ncu CSV of gpu__time_duration.sum,
    dram__bytes_read.sum and dram__bytes_write.sum over whole bench steps: DRAM bytes per call of
    each row (one call per step; the KL and backward rows per call of their block-major pass),
    times `scale` (a capture of a smaller case scaled to the bench workload by the units it
    processes).  Rows not in `only` keep their previous lines."""
    import csv
    import collections
    unit = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    tot = collections.defaultdict(float)
    calls = collections.Counter()      # KL / backward rows: calls counted by their main launch
    firsts = collections.Counter()     # launches of the first kernel of a step
    # several CSVs (comma-separated paths) add up: e.g. one capture per kernel of the same step
    recs = []
    for path in csv_path.split(","):
        # ncu's CSV rows all start with a quote; its "==" messages and the program's own output
        # (when ncu writes to stdout) are skipped
        rows = list(csv.reader(l for l in open(path) if l.startswith('"')))
        hdr = rows[0]
        ki, mi, vi, ui = (hdr.index(c) for c in ("Kernel Name", "Metric Name", "Metric Value",
                                                  "Metric Unit"))
        recs += [(r[ki], r[mi], r[vi], r[ui]) for r in rows[1:]]
    ki, mi, vi, ui = 0, 1, 2, 3
    for r in recs:
        raw = r[ki].split("(")[0]
        name = raw.split("<")[0].split("::")[-1].split()[-1]   # bare kernel name
        if name not in NCU_ROWS:
            continue
        row = NCU_ROWS[name]
        if name == "k_kl_kvouter" and "<" in raw:
            targs = raw[raw.index("<") + 1:raw.rindex(">")].replace(" ", "").split(",")
            if len(targs) >= 3 and targs[2] in ("1", "true"):
                row = "kl_loss_bwd"              # the gradient instantiation (third argument)
        if r[mi] == "gpu__time_duration.sum":
            firsts[name] += 1
            if name in ("k_kl_kvouter", "k_attn_bwd_kvouter"):
                calls[row] += 1
        if r[mi] in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            tot[row] += float(r[vi].replace(",", "")) * unit[r[ui]]
    # one index-branch launch per step (one decode scan when the capture has no prefill)
    steps = firsts["k_index_block_scores"] or firsts["k_decode_block_scores"]
    keep, notes = {}, []
    if os.path.exists(TRAFFIC_FILE):
        for line in open(TRAFFIC_FILE):
            if line.startswith("# capture "):
                notes.append(line.rstrip("\n"))
            elif line.strip() and not line.startswith("#"):
                keep[line.split()[0]] = line.rstrip("\n")
    wrote = []
    for k in ("index_branch", "main_branch", "decode", "kl_loss_fwd", "kl_loss_bwd",
              "sparse_attn_bwd"):
        if k in tot and (only is None or k in only):
            n = calls[k] if k.startswith("kl_") or k == "sparse_attn_bwd" else steps
            keep[k] = "%s %d %s %s" % (k, scale * tot[k] / max(n, 1),
                                       kernel_source_hash(KERNEL_FILES[k]), tag)
            wrote.append(k)
    notes = [x for x in notes if not x.startswith("# capture %s:" % tag)]
    used = {line.split()[3] for line in keep.values() if len(line.split()) >= 4} | {tag}
    notes = [x for x in notes if x.split(":")[0].split()[-1] in used]
    notes.append("# capture %s: %s (rows %s, %d steps, bytes x %g)" % (
        tag, command, ",".join(wrote), steps, scale))
    with open(TRAFFIC_FILE, "w") as f:
        f.write("# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per call of each bench\n"
                "# row, from ncu captures (cold cache) of whole bench steps or of each kernel of one\n"
                "# step; a capture of a smaller case is scaled to the bench workload by the units it\n"
                "# processes (query rows, or the decode batch's algorithmic bytes).\n")
        for n_ in sorted(notes):
            f.write(n_ + "\n")
        f.write("# row  bytes_per_call  source_sha  capture\n")
        for k in ("index_branch", "main_branch", "decode", "kl_loss_fwd", "kl_loss_bwd",
                  "sparse_attn_bwd"):
            if k in keep:
                f.write(keep[k] + "\n")


class Clocks:
    """nvidia-smi samples (200 ms) of this GPU's clocks and throttle reasons."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) == 7:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[3 + k] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][1]) if rows[0][1].replace(".", "").isdigit() else None,
                "samples": len(rows), "reasons": reasons}


# ----------------------------------------------------------------------- workload --

def workload_sizes(pcfg, dcfg, lens):
    N, Hq, Hkv, dh, di, k = pcfg.N, pcfg.H_q, pcfg.H_kv, pcfg.d_h, pcfg.d_idx, pcfg.k
    i = np.arange(N, dtype=np.float64)
    T = np.minimum(i + 1, (k - 1) * 64 + (i % 64) + 1)                # |T_i|
    out = dict(
        F_idx=2.0 * di * Hkv * N * (N + 1) / 2,
        F_main=4.0 * dh * Hq * T.sum(),
        # KL loss: the teacher's scores of the G heads and the student's score per visible token
        F_kl=(2.0 * dh * Hq + 2.0 * di * Hkv) * T.sum(),
    )
    # decode algorithmic bytes: the index-key stream + selected visible K/V + small vectors
    dbytes = 0.0
    for L in (lens if dcfg is not None else []):
        ii = L - 1
        Tt = min(ii + 1, (dcfg.k - 1) * 64 + (ii % 64) + 1)
        dbytes += 2.0 * dcfg.d_idx * L + 2.0 * 2 * dcfg.H_kv * dcfg.d_h * Tt
        dbytes += 2.0 * (2 * dcfg.H_q * dcfg.d_h + dcfg.H_kv * dcfg.d_idx) + 4.0 * dcfg.H_q
    out["decode_bytes"] = dbytes
    return out


def setup(pcfg, dcfg, seed=0):
    msa = __import__("block_sparse_gqa_scores_gb300")
    x = gen.prefill_inputs(pcfg, seed=seed, device="cuda")
    N = pcfg.N
    bufs = dict(
        idx=torch.empty((pcfg.H_kv, N, pcfg.k), dtype=torch.int32, device="cuda"),
        o=torch.empty_like(x["q"]),
        lse=torch.empty((pcfg.H_q, N), dtype=torch.float32, device="cuda"),
        ws=torch.empty(max(16, msa.msa_sparse_attn_fwd_workspace(N, pcfg.H_q, pcfg.H_kv, pcfg.d_h,
                                                                   pcfg.k)),
                       dtype=torch.uint8, device="cuda"),
    )
    if dcfg is None:
        return msa, x, bufs, None, None
    d = gen.decode_inputs(dcfg, seed=seed, device="cuda")
    max_len = dcfg.len_hi
    nws = msa.msa_sparse_decode_workspace(dcfg.S, max_len, dcfg.H_q, dcfg.H_kv, dcfg.d_h,
                                          dcfg.d_idx, dcfg.k)
    dbufs = dict(o=torch.empty_like(d["q"]),
                 lse=torch.empty((dcfg.S, dcfg.H_q), dtype=torch.float32, device="cuda"),
                 idx=torch.empty((dcfg.S, dcfg.H_kv, dcfg.k), dtype=torch.int32, device="cuda"),
                 ws=torch.empty(nws, dtype=torch.uint8, device="cuda"), max_len=max_len)
    return msa, x, bufs, d, dbufs


def bench_config(pcfg, dcfg, world):
    """The workload a bench line measures; both arms report the same object."""
    return {
        "workload": "prefill N=%d" % pcfg.N + (" + decode %d seqs L~U[%d,%d]" % (
            dcfg.S, dcfg.len_lo, dcfg.len_hi) if dcfg is not None else ""),
        "prefill": {"N": pcfg.N, "H_q": pcfg.H_q, "H_kv": pcfg.H_kv, "d_h": pcfg.d_h,
                    "d_idx": pcfg.d_idx, "block": 64, "k": pcfg.k,
                    "hot_blocks": pcfg.hot_blocks, "block_offset_std": pcfg.block_offset_std},
        "decode": {"S": dcfg.S, "len_lo": dcfg.len_lo, "len_hi": dcfg.len_hi, "k": dcfg.k}
        if dcfg is not None else None,
        "l2": "no explicit flush: each step streams Q (1.07 GB), K/V (134 MB each), the "
              "8.8 GB main-branch workspace and the 11.5 GB decode caches, so nothing the "
              "next step reads is still in the 129 MB L2",
        "parallelism": "replicas" if world > 1 else "single",
    }


def run_msa(args, world, rank, local):
    global DEFAULT_WORKLOAD
    DEFAULT_WORKLOAD = args.prefill == "p128k" and not args.prefill_n and args.decode == "decode"
    pcfg = gen.CONFIGS[args.prefill]
    if args.prefill_n:
        pcfg = gen.PrefillConfig(**{**pcfg.__dict__, "N": args.prefill_n})
    dcfg = None if args.decode == "none" else gen.CONFIGS[args.decode]
    if dcfg is not None and args.decode_seqs:
        dcfg = gen.DecodeConfig(**{**dcfg.__dict__, "S": args.decode_seqs})
    DEFAULT_WORKLOAD = DEFAULT_WORKLOAD and not args.decode_seqs
    msa, x, bufs, d, dbufs = setup(pcfg, dcfg, seed=args.seed + rank)
    stream = torch.cuda.current_stream()
    N = pcfg.N

    def prefill():
        # the index branch fused (block scores + top-k, no M), then the main branch
        msa.msa_index_select(x["q_idx"], x["k_idx"], pcfg.k, idx=bufs["idx"])
        ev[1].record(stream)
        msa.msa_sparse_attn_fwd(x["q"], x["k"], x["v"], bufs["idx"], o=bufs["o"], lse=bufs["lse"],
                                ws=bufs["ws"])

    def decode():
        if d is None:
            return
        msa.msa_sparse_decode(d["q"], d["q_idx"], d["k_cache"], d["v_cache"], d["k_idx_cache"],
                              d["cu_seqlens"], dbufs["max_len"], dcfg.k, o=dbufs["o"],
                              lse=dbufs["lse"], idx_out=dbufs["idx"], ws=dbufs["ws"])

    K, W = args.steps, args.warmup
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for _ in range(W):
        ev[0].record(stream)
        prefill()
        ev[2].record(stream)
        decode()
        ev[3].record(stream)
    torch.cuda.synchronize()
    msa.msa_device_status()

    clocks = Clocks(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(K):
        ev = evs[s]
        ev[0].record(stream)
        prefill()
        ev[2].record(stream)
        decode()
        ev[3].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    msa.msa_device_status()

    per = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(3)] for e in evs])   # ms
    t_index, t_attn, t_decode = per.mean(axis=0)
    t_prefill_total = max_over_ranks(float(per[:, :2].sum()), world)   # ms over K steps
    t_decode_total = max_over_ranks(float(per[:, 2].sum()), world)
    t_all = max_over_ranks(t_start.elapsed_time(t_end), world)

    sizes = workload_sizes(pcfg, dcfg, d["meta"]["lens"] if d else [])
    pk = peaks()
    kern = []

    def add(name, ms, bound, work, unit, traffic=None):
        kern.append(roofline_row(name, ms, bound, work, unit, pk, traffic))

    add("index_branch", t_index, "tensor", sizes["F_idx"], "TFLOP/s",
        ncu_traffic("index_branch"))
    add("main_branch", t_attn, "tensor", sizes["F_main"], "TFLOP/s", ncu_traffic("main_branch"))
    if d is not None:
        add("decode (%d kernels)" % DECODE_LAUNCHES, t_decode, "hbm", sizes["decode_bytes"],
            "GB/s", ncu_traffic("decode"))
    dom = max(kern, key=lambda r: r["ms"])

    value = world * N * K / (t_prefill_total * 1e-3)
    dec_value = world * dcfg.S * K / (t_decode_total * 1e-3) if d is not None else None
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(t_all / K, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(pcfg, dcfg, world),
        "ms_prefill": round(t_prefill_total / K, 4),
        "ms_decode": round(t_decode_total / K, 4),
        "decode": {"value": round(dec_value, 1), "unit": "tokens/s",
                   "ms": round(t_decode_total / K, 4),
                   "mean_len": float(np.mean(d["meta"]["lens"]))} if d is not None else None,
        "kernels": kern,
        "roofline": {k_: dom[k_] for k_ in ("kernel", "bound", "achieved", "peak", "unit", "frac",
                                             "traffic", "peak_source")
                     if k_ in dom} | ({"frac_of_sustained": dom["frac_of_sustained"]}
                                      if "frac_of_sustained" in dom else {}),
        "clocks": clk,
        "gpu_launches": (1 + ATTN_LAUNCHES_PER_CHUNK * (-(-N // ATTN_CHUNK_ROWS)) +
                         (DECODE_LAUNCHES if d is not None else 0)) * K,
    }
    if not args.no_kl:
        line["kl_loss_fwd"] = time_kl(msa, pcfg, x, bufs, K, sizes, pk, world)
    if not args.no_bwd:
        line["sparse_attn_bwd"] = time_bwd(msa, pcfg, x, bufs, K, sizes, pk, world)
    if DEFAULT_WORKLOAD and not args.no_extra_prefill:
        # the other two prefill lengths of the workload set, each on its own inputs
        for key, name in (("prefill_32k", "p32k"), ("prefill_1m", "p1m")):
            line[key] = time_prefill_only(msa, gen.CONFIGS[name], bufs, K, pk, world,
                                          seed=args.seed + rank)
    if d is not None and not args.no_paged:
        line["decode_paged"] = time_decode_paged(msa, dcfg, d, dbufs, K, sizes, pk, world)
    if not args.no_varlen and pcfg.k <= 32:
        line["prefill_varlen"] = time_varlen(msa, pcfg, x, bufs, K, world)
    if not args.no_e2e:
        line["e2e"] = e2e_prefill(msa, pcfg, x, bufs, K, W, world)
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(pcfg, x, args.cpu_seconds, args.seed)
    return line


def roofline_row(name, ms, bound, work, unit, pk, traffic=None):
    """One kernel row: achieved = algorithmic work / measured time.  Tensor-bound rows are
    divided by the burst bf16 peak (these rows run in sub-second loops at full clocks); the
    fraction of the sustained (power-capped) figure is given beside it."""
    achieved = work / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
    row = {"kernel": name, "ms": round(ms, 4), "bound": bound, "achieved": round(achieved, 2),
           "unit": unit, "traffic": traffic, "algorithmic": work}
    if unit == "TFLOP/s":
        row.update(peak=pk["bf16"], frac=round(achieved / pk["bf16"], 4),
                   frac_of_sustained=round(achieved / pk["bf16_sust"], 4),
                   peak_source="%s (bf16 burst)" % pk["src"])
    else:
        row.update(peak=pk["hbm"], frac=round(achieved / pk["hbm"], 4),
                   peak_source="%s (HBM copy)" % pk["src"])
    return row


def time_prefill_only(msa, pcfg, bufs, K, pk, world, seed=0):
    """Prefill alone (fused index branch, then the main branch) on a workload of its own, timed
    apart from the step: K calls after 3 warm-up calls, per-call CUDA events around each of the
    two calls.  The main branch reuses the step's workspace (sized for any N > 65536)."""
    x = gen.prefill_inputs(pcfg, seed=seed, device="cuda")
    N = pcfg.N
    idx = torch.empty((pcfg.H_kv, N, pcfg.k), dtype=torch.int32, device="cuda")
    o = torch.empty_like(x["q"])
    lse = torch.empty((pcfg.H_q, N), dtype=torch.float32, device="cuda")
    need = msa.msa_sparse_attn_fwd_workspace(N, pcfg.H_q, pcfg.H_kv, pcfg.d_h, pcfg.k)
    ws = bufs["ws"] if bufs["ws"].numel() >= need else torch.empty(need, dtype=torch.uint8,
                                                                   device="cuda")
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]

    def call(e=None):
        if e is not None:
            e[0].record(stream)
        msa.msa_index_select(x["q_idx"], x["k_idx"], pcfg.k, idx=idx)
        if e is not None:
            e[1].record(stream)
        msa.msa_sparse_attn_fwd(x["q"], x["k"], x["v"], idx, o=o, lse=lse, ws=ws)
        if e is not None:
            e[2].record(stream)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    for s in range(K):
        call(ev[s])
    torch.cuda.synchronize()
    msa.msa_device_status()
    t_i = max_over_ranks(float(np.mean([e[0].elapsed_time(e[1]) for e in ev])), world)
    t_a = max_over_ranks(float(np.mean([e[1].elapsed_time(e[2]) for e in ev])), world)
    sz = workload_sizes(pcfg, None, [])
    del x, o, idx, lse
    return {"N": N, "value": round(world * N / ((t_i + t_a) * 1e-3), 1), "unit": "tokens/s",
            "ms": round(t_i + t_a, 4),
            "kernels": [roofline_row("index_branch", t_i, "tensor", sz["F_idx"], "TFLOP/s", pk),
                        roofline_row("main_branch", t_a, "tensor", sz["F_main"], "TFLOP/s", pk)]}


# the main-branch backward: ordered bucketing (2 memsets, count, scan, bases, scatter), piece
# offsets, delta, the block-major gradient pass, the dQ merge and the dK/dV merge
BWD_LAUNCHES = 9


def time_bwd(msa, pcfg, x, bufs, K, sizes, pk, world):
    """The main-branch backward (dQ, dK, dV) on the last step's selection, O and LSE with a seeded
    upstream gradient, timed apart from the step: K calls after 3 warm-up calls.  Work counted:
    per visible selected token and head the five d_h-long products S, dP, dV, dK and dQ, i.e.
    2.5 times the forward's."""
    N = pcfg.N
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    d_o = torch.randn(x["q"].shape, generator=g, device="cuda").to(torch.bfloat16)
    dq = torch.empty(x["q"].shape, dtype=torch.float32, device="cuda")
    dk = torch.empty(x["k"].shape, dtype=torch.float32, device="cuda")
    dv = torch.empty(x["v"].shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(msa.msa_sparse_attn_bwd_workspace(N, pcfg.H_q, pcfg.H_kv, pcfg.d_h, pcfg.k),
                     dtype=torch.uint8, device="cuda")

    def call():
        msa.msa_sparse_attn_bwd(x["q"], x["k"], x["v"], bufs["idx"], bufs["o"], bufs["lse"], d_o,
                                dq=dq, dk=dk, dv=dv, ws=ws)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    evs[0].record(stream)
    for s in range(K):
        call()
        evs[s + 1].record(stream)
    torch.cuda.synchronize()
    msa.msa_device_status()
    ms = max_over_ranks(float(np.mean([evs[s].elapsed_time(evs[s + 1]) for s in range(K)])), world)
    finite = bool(torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all())
    del ws, dq, dk, dv, d_o
    return {"ms": round(ms, 4), "value": round(world * N / (ms * 1e-3), 1), "unit": "tokens/s",
            "gpu_launches_per_call": BWD_LAUNCHES, "finite": finite,
            "roofline": roofline_row("sparse_attn_bwd", ms, "tensor", 2.5 * sizes["F_main"],
                                     "TFLOP/s", pk, ncu_traffic("sparse_attn_bwd"))}


def time_kl(msa, pcfg, x, bufs, K, sizes, pk, world):
    """The KL alignment loss forward (the training-side consumer of the forward's LSE) on the
    last step's selection and LSE, timed apart from the step: K calls after 3 warm-up calls."""
    N = pcfg.N
    kl = torch.empty((pcfg.H_kv, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(msa.msa_kl_loss_fwd_workspace(N, pcfg.H_kv, pcfg.k), dtype=torch.uint8,
                     device="cuda")

    def call():
        msa.msa_kl_loss_fwd(x["q"], x["k"], x["q_idx"], x["k_idx"], bufs["idx"], bufs["lse"],
                            kl=kl, ws=ws)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    evs[0].record(stream)
    for s in range(K):
        call()
        evs[s + 1].record(stream)
    torch.cuda.synchronize()
    msa.msa_device_status()
    ms = max_over_ranks(float(np.mean([evs[s].elapsed_time(evs[s + 1]) for s in range(K)])), world)
    # the index-branch gradient of the loss (teacher fixed), on the same inputs, g = 1 per row
    lse_idx = torch.empty((pcfg.H_kv, N), dtype=torch.float32, device="cuda")
    psum = torch.empty_like(lse_idx)
    msa.msa_kl_loss_fwd(x["q"], x["k"], x["q_idx"], x["k_idx"], bufs["idx"], bufs["lse"], kl=kl,
                        ws=ws, lse_idx=lse_idx, p_sum=psum)
    del ws
    g = torch.ones_like(lse_idx)
    dq = torch.empty((N, pcfg.H_kv, pcfg.d_idx), dtype=torch.float32, device="cuda")
    dk = torch.empty((N, pcfg.d_idx), dtype=torch.float32, device="cuda")
    wsb = torch.empty(msa.msa_kl_loss_bwd_workspace(N, pcfg.H_kv, pcfg.d_idx, pcfg.k),
                      dtype=torch.uint8, device="cuda")

    def bwd():
        msa.msa_kl_loss_bwd(x["q"], x["k"], x["q_idx"], x["k_idx"], bufs["idx"], bufs["lse"],
                            lse_idx, psum, g, dq_idx=dq, dk_idx=dk, ws=wsb)

    for _ in range(3):
        bwd()
    torch.cuda.synchronize()
    evb = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    evb[0].record(stream)
    for s in range(K):
        bwd()
        evb[s + 1].record(stream)
    torch.cuda.synchronize()
    msa.msa_device_status()
    del wsb
    ms_b = max_over_ranks(float(np.mean([evb[s].elapsed_time(evb[s + 1]) for s in range(K)])),
                          world)
    return {"ms": round(ms, 4), "value": round(world * N / (ms * 1e-3), 1), "unit": "tokens/s",
            "backward_index_branch": {"ms": round(ms_b, 4),
                                      "value": round(world * N / (ms_b * 1e-3), 1),
                                      "unit": "tokens/s", "gpu_launches_per_call": KLB_LAUNCHES,
                                      "traffic": ncu_traffic("kl_loss_bwd")},
            "mean_kl": round(float(kl.mean()), 6), "gpu_launches_per_call": KL_LAUNCHES,
            "roofline": roofline_row("kl_loss_fwd", ms, "tensor", sizes["F_kl"], "TFLOP/s", pk,
                                     ncu_traffic("kl_loss_fwd"))}


def time_decode_paged(msa, dcfg, d, dbufs, K, sizes, pk, world):
    """Decode of the same batch from a paged cache (the tokens in shuffled 64-token pages),
    timed apart from the step: K calls after 3 warm-up calls."""
    kp, vp, kip, pt, sl = gen.to_pages(d, seed=1)
    max_len = min(dbufs["max_len"], 64 * pt.shape[1])
    o, lse = torch.empty_like(dbufs["o"]), torch.empty_like(dbufs["lse"])
    idx = torch.empty_like(dbufs["idx"])

    def call():
        msa.msa_sparse_decode_paged(d["q"], d["q_idx"], kp, vp, kip, pt, sl, max_len, dcfg.k,
                                    o=o, lse=lse, idx_out=idx, ws=dbufs["ws"])

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    evs[0].record(stream)
    for s in range(K):
        call()
        evs[s + 1].record(stream)
    torch.cuda.synchronize()
    msa.msa_device_status()
    same = bool(torch.equal(o, dbufs["o"]) and torch.equal(idx, dbufs["idx"]))
    del kp, vp, kip
    ms = max_over_ranks(float(np.mean([evs[s].elapsed_time(evs[s + 1]) for s in range(K)])), world)
    achieved = sizes["decode_bytes"] / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 4), "value": round(world * dcfg.S / (ms * 1e-3), 1),
            "unit": "tokens/s", "equals_packed": same, "gpu_launches_per_call": DECODE_LAUNCHES,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": pk["hbm"],
                         "unit": "GB/s", "frac": round(achieved / pk["hbm"], 4),
                         "algorithmic": sizes["decode_bytes"]}}


VARLEN_LENS = (65536, 32768, 16384, 8192, 4096, 2048, 1024, 512, 256, 256)
VARLEN_UNIFORM = (64, 2048)       # a batch of many equal short sequences (count, length)


def time_varlen(msa, pcfg, x, bufs, K, world):
    """Varlen prefill of the same N tokens cut into independent sequences of mixed lengths
    (VARLEN_LENS scaled to N), timed apart from the step: K calls after 3 warm-up calls.  It
    overwrites the step's output buffers, so it runs after every other use of them."""
    N = pcfg.N
    lens = [max(1, L * N // 131072) for L in VARLEN_LENS]
    lens[0] += N - sum(lens)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.tensor(lens), 0)
    # one workspace for both batches (the virtual rows of a batch can outnumber its tokens)
    cnt, ln = VARLEN_UNIFORM
    cu2 = torch.arange(cnt + 1, dtype=torch.int64) * ln
    nws = max(msa.msa_prefill_varlen_workspace(c, pcfg.H_q, pcfg.H_kv, pcfg.d_h, pcfg.k)
              for c in (cu, cu2))
    ws = bufs["ws"] if nws <= bufs["ws"].numel() else torch.empty(nws, dtype=torch.uint8,
                                                                     device="cuda")

    def call():
        msa.msa_prefill_varlen(x["q"], x["k"], x["v"], x["q_idx"], x["k_idx"], cu, pcfg.k,
                               o=bufs["o"], lse=bufs["lse"].view(-1), idx=bufs["idx"].view(-1),
                               ws=ws)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    evs[0].record(stream)
    for s in range(K):
        call()
        evs[s + 1].record(stream)
    torch.cuda.synchronize()
    msa.msa_device_status()
    ms = max_over_ranks(float(np.mean([evs[s].elapsed_time(evs[s + 1]) for s in range(K)])), world)
    out = {"ms": round(ms, 4), "value": round(world * N / (ms * 1e-3), 1), "unit": "tokens/s",
           "sequences": lens}
    # many equal short sequences: launch count per sequence matters most here
    if cnt * ln <= N:
        T = cnt * ln

        def call2():
            msa.msa_prefill_varlen(x["q"][:T], x["k"][:T], x["v"][:T], x["q_idx"][:T],
                                   x["k_idx"][:T], cu2, pcfg.k, o=bufs["o"][:T],
                                   lse=bufs["lse"].view(-1)[:T * pcfg.H_q],
                                   idx=bufs["idx"].view(-1)[:T * pcfg.H_kv * pcfg.k], ws=ws)

        for _ in range(3):
            call2()
        torch.cuda.synchronize()
        ev2 = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
        ev2[0].record(stream)
        for s in range(K):
            call2()
            ev2[s + 1].record(stream)
        torch.cuda.synchronize()
        msa.msa_device_status()
        ms2 = max_over_ranks(float(np.mean([ev2[s].elapsed_time(ev2[s + 1]) for s in range(K)])),
                             world)
        out["uniform"] = {"sequences": cnt, "length": ln, "ms": round(ms2, 4),
                          "value": round(world * T / (ms2 * 1e-3), 1), "unit": "tokens/s"}
    return out


def e2e_prefill(msa, pcfg, x, bufs, K, W, world):
    """Prefill through the public calls with host (pinned) inputs and outputs: every step copies
    its Q, K, V, Q_idx, K_idx host -> device, runs the two calls, and reads O and LSE back to the
    host, all inside the timed region.  The steps are pipelined as a serving loop would run
    them: two device buffer sets, the host -> device copies on one stream and the device -> host
    reads on another, so step s+1's inputs and step s-1's results move while step s computes
    (each stream's order and the events keep every copy after the step it belongs to).  Q_idx
    and K_idx are copied first and the index branch waits only for them, so in the first step
    the Q, K and V copies run under the index branch."""
    # the index branch's inputs first: it starts on them while Q, K and V are still copying
    names = ["q_idx", "k_idx", "q", "k", "v"]
    host = {n: torch.empty(x[n].shape, dtype=x[n].dtype, pin_memory=True) for n in names}
    for n in names:
        host[n].copy_(x[n])
    dev = [{n: torch.empty_like(x[n]) for n in names} for _ in range(2)]
    outs = [(torch.empty_like(bufs["o"]), torch.empty_like(bufs["lse"])) for _ in range(2)]
    o_h = torch.empty(bufs["o"].shape, dtype=bufs["o"].dtype, pin_memory=True)
    l_h = torch.empty(bufs["lse"].shape, dtype=bufs["lse"].dtype, pin_memory=True)
    N = pcfg.N
    comp = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    idx_ready = [ev(), ev()]     # Q_idx and K_idx of the buffer set copied
    in_ready = [ev(), ev()]      # Q, K and V of the buffer set copied
    in_free = [ev(), ev()]       # the step that read the buffer set's inputs is done
    out_ready = [ev(), ev()]     # the step's outputs written
    out_free = [ev(), ev()]      # the outputs read back to the host
    started = [False, False]

    def step(i):
        j = i & 1
        with torch.cuda.stream(h2d_s):
            if started[j]:
                h2d_s.wait_event(in_free[j])
            for n in names:
                dev[j][n].copy_(host[n], non_blocking=True)
                if n == "k_idx":
                    idx_ready[j].record(h2d_s)
            in_ready[j].record(h2d_s)
        comp.wait_event(idx_ready[j])
        if started[j]:
            comp.wait_event(out_free[j])
        idx = msa.msa_index_select(dev[j]["q_idx"], dev[j]["k_idx"], pcfg.k, idx=bufs["idx"])
        comp.wait_event(in_ready[j])
        msa.msa_sparse_attn_fwd(dev[j]["q"], dev[j]["k"], dev[j]["v"], idx, o=outs[j][0],
                                lse=outs[j][1], ws=bufs["ws"])
        in_free[j].record(comp)
        out_ready[j].record(comp)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(out_ready[j])
            o_h.copy_(outs[j][0], non_blocking=True)
            l_h.copy_(outs[j][1], non_blocking=True)
            out_free[j].record(d2h_s)
        started[j] = True

    def run(n0, n):
        for i in range(n0, n0 + n):
            step(i)
        # the step sequence ends once the last reads are on the host
        for j in range(2):
            if started[j]:
                comp.wait_event(out_free[j])

    run(0, W)
    torch.cuda.synchronize()
    # the host link on its own (outside the timed region): one input copy each way, for reading
    # the e2e figure against the device time
    link = {}
    for name, dst, src in (("h2d_gbs", dev[0]["k"], host["k"]), ("d2h_gbs", o_h, outs[0][0])):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        dst.copy_(src, non_blocking=True)
        e1.record(comp)
        torch.cuda.synchronize()
        link[name] = round(src.numel() * src.element_size() / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    h2d_s.wait_event(a)
    d2h_s.wait_event(a)
    run(W, K)
    b.record(comp)
    torch.cuda.synchronize()
    t = max_over_ranks(a.elapsed_time(b), world)
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = o_h.numel() * o_h.element_size() + l_h.numel() * l_h.element_size()
    del dev, host, outs
    return {"value": round(world * N * K / (t * 1e-3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(t / K, 4), "copies": "pipelined over steps", **link}


def cpu_sample_rows(N, n, seed):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(N, size=n, replace=False)).astype(np.int64)


def oracle_rows_rate(pcfg, xh, seconds, seed, max_rows=4096, batch=16):
    """Times the oracle's whole prefill path on uniformly sampled query rows until about
    `seconds` of CPU work; returns (rows/s, rows, threads)."""
    import oracle
    oracle.build()
    rows_all = cpu_sample_rows(pcfg.N, max_rows, seed)
    done, t = 0, 0.0
    while t < seconds and done < max_rows:
        rows = rows_all[done:done + batch]
        qr = np.ascontiguousarray(xh["q"][rows])
        qir = np.ascontiguousarray(xh["q_idx"][rows])
        t0 = time.perf_counter()
        oracle.prefill(qr, xh["k"], xh["v"], qir, xh["k_idx"], pcfg.k, rows=rows, compact=True)
        t += time.perf_counter() - t0
        done += len(rows)
    return done / t, done, oracle.get_threads()


def host_bits(x, names=("k", "v", "k_idx")):
    out = {n: gen.to_bits(x[n]) for n in names}
    return out


def cpu_baseline(pcfg, x, seconds, seed):
    xh = host_bits(x)
    xh["q"] = gen.to_bits(x["q"])
    xh["q_idx"] = gen.to_bits(x["q_idx"])
    rate, rows, cores = oracle_rows_rate(pcfg, xh, seconds, seed)
    return {"value": round(rate, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "%d uniformly sampled query rows of the N=%d prefill workload, whole path "
                      "(causal index scores, selection, main branch), fp64" % (rows, pcfg.N)}


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm, on bounded samples of the prefill workload."""
    if rank != 0:
        return None
    pcfg = gen.CONFIGS[args.prefill]
    if args.prefill_n:
        pcfg = gen.PrefillConfig(**{**pcfg.__dict__, "N": args.prefill_n})
    dcfg = None if args.decode == "none" else gen.CONFIGS[args.decode]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x = gen.prefill_inputs(pcfg, seed=args.seed, device=dev)
    xh = host_bits(x, ("q", "k", "v", "q_idx", "k_idx"))
    del x
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_rows_rate(pcfg, xh, per_step / 4, args.seed, batch=8)
    rates, total_rows = [], 0
    t0 = time.perf_counter()
    for s in range(args.steps):
        rate, rows, cores = oracle_rows_rate(pcfg, xh, per_step, args.seed + 1 + s, batch=8)
        rates.append(rate)
        total_rows += rows
    elapsed = time.perf_counter() - t0
    value = float(np.mean(rates))
    return {"metric": METRIC, "impl": "reference", "value": round(value, 3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * elapsed / args.steps, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(pcfg, dcfg, world),
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores,
                             "kind": "oracle",
                             "sample": "%d uniformly sampled query rows per run of the N=%d "
                                       "prefill workload, whole prefill path, fp64 (the metric "
                                       "is prefill tokens/s; decode is not timed on this arm)" % (
                                           total_rows // args.steps, pcfg.N)},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["msa", "reference"], default="msa")
    ap.add_argument("--prefill", default="p128k")
    ap.add_argument("--prefill-n", type=int, default=None,
                    help="override the prefill length (same head layout and structure)")
    ap.add_argument("--decode", default="decode", help="decode workload, or 'none'")
    ap.add_argument("--decode-seqs", type=int, default=None,
                    help="override the decode batch size (same length range)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-kl", action="store_true", help="skip the KL loss forward measurement")
    ap.add_argument("--no-paged", action="store_true",
                    help="skip the paged-cache decode measurement")
    ap.add_argument("--no-varlen", action="store_true",
                    help="skip the varlen (batched) prefill measurement")
    ap.add_argument("--no-bwd", action="store_true",
                    help="skip the main-branch backward measurement")
    ap.add_argument("--no-extra-prefill", action="store_true",
                    help="skip the 32K and 1M prefill measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--write-traffic", metavar="NCU_CSV",
                    help="write profiles/traffic.txt from ncu CSVs (comma-separated) that "
                         "together cover whole steps, and exit")
    ap.add_argument("--traffic-command", default="",
                    help="the command the ncu CSV was captured on (recorded in the file)")
    ap.add_argument("--traffic-scale", type=float, default=1.0,
                    help="factor from the captured case to the bench workload (query rows)")
    ap.add_argument("--traffic-rows", default="",
                    help="comma-separated rows to update (default: every row in the capture)")
    ap.add_argument("--traffic-tag", default="A", help="capture label recorded per row")
    args = ap.parse_args()
    if args.write_traffic:
        write_traffic(args.write_traffic, args.traffic_command, args.traffic_scale,
                      set(args.traffic_rows.split(",")) if args.traffic_rows else None,
                      args.traffic_tag)
        return
    if args.warmup < 3 and args.impl == "msa":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_msa(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
