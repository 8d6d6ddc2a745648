#!/usr/bin/env python3
"""Fused linear cross-entropy forward+backward throughput on GB300.

One step = one flce_fwd_bwd call (logits GEMM + online LSE, merge, then per
vocabulary chunk the dZ recompute, dW and dX GEMMs, and the dX conversion)
over one batch of N tokens of the chosen synthetic workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0.  ``value`` is tokens/s over all ranks with
inputs resident in HBM; ``e2e`` is the same metric with the inputs (X, W,
labels) copied from pinned host memory and the step's result (the loss) read
back inside the timed region, and ``e2e_all_outputs`` the same with every
output (loss, lse, dX, dW) read back.  With N > 1 every rank runs its own batch (weak scaling, no
collective on the data path).  ``--impl reference`` times the fp64 CPU oracle
on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused fwd+bwd tokens/s and TFLOP/s (% of BF16 tensor roofline), 1×GB300"
DEFAULT_WORKLOAD = "llama3_n8192"


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=150)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--shape", default=None,
                    help="N,H,V override of the workload's shape (same input recipe); "
                         "for small profiler captures")
    ap.add_argument("--vocab-chunk", type=int, default=0,
                    help="vocabulary columns per backward chunk (0 = automatic)")
    ap.add_argument("--cpu-baseline-rows", type=int, default=1024,
                    help="token rows of the oracle sample timed on the host (0 = skip)")
    ap.add_argument("--reference-rows", type=int, default=128,
                    help="token rows per oracle step of --impl reference")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--copy-streams", type=int, default=4,
                    help="end-to-end leg: copy streams per direction (large copies are split)")
    ap.add_argument("--summarize-traffic", metavar="NCU_CSV", default=None,
                    help="write profiles/traffic_<workload>.txt from an ncu --csv capture of "
                         "dram__bytes_read.sum / dram__bytes_write.sum, then exit; with "
                         "--shape, the capture ran at that reduced shape (see summarize_traffic)")
    ap.add_argument("--l2-hints", action="store_true",
                    help="evict_last L2 policy for the operand re-read on every wave of tiles")
    ap.add_argument("--vocab-shards", type=int, default=0,
                    help="time the vocabulary-parallel layout with this many shards run one "
                         "after another on the GPU (stack / sum stand in for the exchange)")
    ap.add_argument("--grad-filter", type=float, default=0.0,
                    help="gradient filtering threshold eps_f (e.g. 2**-12; 0 = exact)")
    ap.add_argument("--skip-ignored", action="store_true",
                    help="skip token blocks whose labels are all ignore_index")
    ap.add_argument("--z-loss", type=float, default=0.0,
                    help="z-loss weight alpha (adds alpha * lse^2 per valid token)")
    ap.add_argument("--multicast", type=int, default=None, choices=(0, 1),
                    help="operand multicast between CTA pairs in 4-CTA clusters (1) or plain "
                         "CTA pairs (0); default: the library's default")
    ap.add_argument("--single-cta", action="store_true",
                    help="128x256 single-CTA tiles instead of 256x256 CTA-pair tiles")
    ap.add_argument("--clocks-dir", default=None,
                    help="directory for the raw nvidia-smi clock samples (default: temp dir)")
    ap.add_argument("--merge", type=int, nargs="?", const=1, default=None, choices=(0, 1, 2),
                    help="backward layout: 0 three launches per vocabulary chunk; 1 (bare "
                         "--merge) one merged dW(c) + dX(c) + dZ(c+1) launch per chunk (two dZ "
                         "buffers); 2 dZ(c) alone, then one merged dW(c) + dX(c) launch; "
                         "default: the library's default layout")
    return ap.parse_args()


KERNEL_SOURCES = ("gemm_core.cuh", "bwd_fused.cuh", "ptx.cuh", "aux_kernels.cuh", "flce_api.cu")
KIND_BY_EPI = {("0", None): "fwd_logits_lse", ("1", None): "bwd_dz_recompute",
               ("2", "1"): "bwd_dw_gemm", ("2", "0"): "bwd_dx_gemm"}


def kernel_source_hash() -> str:
    """SHA-256 of the CUDA sources the GEMM kinds are built from."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "linear_cross_entropy_logit_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def traffic_path(workload: str) -> str:
    return os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")


def summarize_traffic(csv_path: str, workload: str, shape=None) -> None:
    """Per-kind DRAM bytes per launch from an ncu CSV (mangled kernel names).

    Each kind's LAST captured launch is kept (a capture of the first backward
    chunks ends on a full-width chunk whose dX launch reduce-adds, as all but
    the first chunk's do).  ``shape`` = (N, H, V) of a reduced capture with
    the workload's N and H and the same chunk width: the dZ, dW and dX launches
    of a full-width chunk then have the full-size shape and are kept as they
    are; the forward's units grow with V (W is streamed once per row band), so
    its bytes are scaled by V_full / V_capture."""
    import csv
    import re
    per = {}
    with open(csv_path) as fh:
        rows = list(csv.DictReader(l for l in fh if not l.startswith("==")))
    for r in rows:
        name = r["Kernel Name"]
        m = (re.search(r"EpiE(\d)ELb(\d)ELb(\d)", name)
             or re.search(r"gemm_(?:pair_|quad_)?kernel<(\d), (\d), (\d), \d+(?:, \d)?>", name))
        if "bwd_fused_kernel" in name:
            kind = "bwd_merged"
        elif m:
            kind = KIND_BY_EPI.get((m.group(1), None)) or KIND_BY_EPI[(m.group(1), m.group(2))]
        else:
            continue
        d = per.setdefault(kind, {"last": None, "n": 0, "read": {}, "write": {}})
        lid = int(r["ID"])
        if d["last"] != lid:
            d["n"] += 1
            d["last"] = lid
        scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}.get(r["Metric Unit"], None)
        if scale is None:
            continue
        v = float(r["Metric Value"].replace(",", "")) * scale
        if r["Metric Name"] == "dram__bytes_read.sum":
            d["read"][lid] = v
        elif r["Metric Name"] == "dram__bytes_write.sum":
            d["write"][lid] = v
    note = "full size"
    fwd_scale = 1.0
    if shape is not None:
        from linear_cross_entropy_logit_gb300 import inputs as I
        full = I.CONFIGS[workload]
        N, H, V = shape
        if (N, H) != (full.N, full.H):
            raise ValueError("a reduced capture must keep the workload's N and H")
        fwd_scale = full.V / V
        note = (f"captured at N={N} H={H} V={V}; forward scaled by {fwd_scale:.4f}, "
                "backward launches of a full-width chunk as captured")
    lines = [f"# DRAM bytes per launch, {workload}, from {os.path.basename(csv_path)} ({note})",
             f"# source_sha256 {kernel_source_hash()}",
             "# kind launches_captured read_bytes_per_launch write_bytes_per_launch"]
    for kind, d in sorted(per.items()):
        k = d["last"]
        f = fwd_scale if kind == "fwd_logits_lse" else 1.0
        lines.append(f"{kind} {d['n']} {d['read'].get(k, 0.0) * f:.0f} "
                     f"{d['write'].get(k, 0.0) * f:.0f}")
    with open(traffic_path(workload), "w") as fh:
        fh.write("\n".join(lines) + "\n")
    print("\n".join(lines))


def load_traffic(workload: str):
    """{kind: bytes per launch} if the capture matches the current kernel source."""
    try:
        with open(traffic_path(workload)) as fh:
            lines = fh.read().splitlines()
    except OSError:
        return None
    sha = next((l.split()[2] for l in lines if l.startswith("# source_sha256")), None)
    if sha != kernel_source_hash():
        return None
    out = {}
    for l in lines:
        if l and not l.startswith("#"):
            kind, n, rd, wr = l.split()
            out[kind] = float(rd) + float(wr)
    return out


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {"bf16_burst": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0,
                "source": "fallback"}


# The sustained bf16 figure is a cuBLAS GEMM run back to back for seconds
# under the power cap; the burst figure a short best-of-ten.  A timed loop at
# least this long has settled under the cap like the sustained loop, so it is
# stated against that figure; a shorter one against the burst figure.
SUSTAINED_LOOP_S = 2.0


def peak_choice(pk: dict, wall_s: float):
    """(name, TFLOP/s, reason) of the bf16 peak a timed loop of wall_s seconds
    is stated against."""
    if wall_s >= SUSTAINED_LOOP_S:
        return ("sustained", pk["bf16_sustained"],
                f"at least {SUSTAINED_LOOP_S:g} s of back-to-back work under the power cap, "
                "like the sustained figure's own loop")
    return ("burst", pk["bf16_burst"],
            f"shorter than {SUSTAINED_LOOP_S:g} s, so the clock has not settled under the cap")


# ----------------------------------------------------------------------------
# Clock sampling during the timed region
# ----------------------------------------------------------------------------
CLOCK_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                "clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: str, out_dir: str | None = None):
        import tempfile
        self.proc = None
        self.path = os.path.join(out_dir or tempfile.gettempdir(),
                                 f"clocks_bench_{os.getpid()}.csv")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", gpu_index], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) != 7:
                    continue
                try:
                    rows.append((float(parts[0]), float(parts[1]), parts[2], parts[3:]))
                except ValueError:
                    continue
        if not rows:
            return None
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "samples": len(rows),
                "reasons": reasons}


# ----------------------------------------------------------------------------
# Reference arm: the fp64 oracle on the host cores
# ----------------------------------------------------------------------------
def oracle_sample(wl, rows: int, z_loss: float = 0.0):
    """The oracle's fused forward+backward on the first ``rows`` tokens."""
    from oracle import flce_oracle as O
    r = min(rows, wl.N)
    t0 = time.perf_counter()
    O.fwd_bwd(wl.x[:r], wl.w, wl.labels[:r], wl.spec.ignore_index, wl.spec.smoothing,
              wl.spec.reduction, z_loss=z_loss)
    return r, time.perf_counter() - t0


def run_reference(args, rank: int):
    from linear_cross_entropy_logit_gb300 import inputs as I
    if rank != 0:
        return
    spec = workload_spec(args)
    wl = I.make_workload(spec, seed=args.seed)
    for _ in range(args.warmup):
        oracle_sample(wl, args.reference_rows, args.z_loss)
    total_rows, total_s = 0, 0.0
    for _ in range(args.steps):
        r, dt = oracle_sample(wl, args.reference_rows, args.z_loss)
        total_rows += r
        total_s += dt
    value = total_rows / total_s
    cores = host_cores()
    sample = (f"first {min(args.reference_rows, wl.N)} of {wl.N} tokens per step, full V and H, "
              f"fp64 oracle forward+backward (numpy float64 matmul)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": line_config(spec, args, args.gpus),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_spec(args):
    import dataclasses
    from linear_cross_entropy_logit_gb300 import inputs as I
    spec = I.CONFIGS[args.workload]
    if args.shape:
        N, H, V = (int(v) for v in args.shape.split(","))
        spec = dataclasses.replace(spec, name=f"{spec.name}@{N}x{H}x{V}", N=N, H=H, V=V,
                                   n_ignore=min(spec.n_ignore, N),
                                   n_scaled_w_rows=min(spec.n_scaled_w_rows, V))
    return spec


def kind_flops(B, N, H, V, args, merged):
    """Algorithmic FLOP per step of each profiled kernel kind.

    Forward, dZ recompute, dW and dX each contract 2*N*V*H per step.  With the
    merged dW(c) + dX(c) + dZ(c+1) launches (merged = 1) the dZ kind runs only
    chunk 0 of each backward call (2*N*w0*H) and the merged kind the rest of
    the three backward contractions (6*N*V*H minus that); with merged dW(c) +
    dX(c) launches (merged = 2) the merged kind does 4*N*V*H."""
    calls = [V]
    if args.vocab_shards > 1:
        P = args.vocab_shards
        bounds = [round(V * i / P / 256) * 256 for i in range(P)] + [V]
        calls = [b1 - b0 for b0, b1 in zip(bounds, bounds[1:])]
    full = 2.0 * N * V * H
    out = {"fwd_logits_lse": full, "bwd_dz_recompute": full, "bwd_dw_gemm": full,
           "bwd_dx_gemm": full, "bwd_merged": 0.0}
    if merged == 2:
        out["bwd_merged"] = 2.0 * full
    elif merged:
        dz0 = sum(2.0 * N * min(B.flce_vocab_chunk(N, H, v), v) * H for v in calls)
        out["bwd_dz_recompute"] = dz0
        out["bwd_merged"] = 3.0 * full - dz0
    return out


def backward_layout(mode, args) -> str:
    """What the backward of this run launches per vocabulary chunk."""
    if mode == 0 or args.single_cta or args.skip_ignored or args.grad_filter or args.l2_hints:
        return "three launches per vocabulary chunk"
    if mode == 1:
        return "merged dW(c) + dX(c) + dZ(c+1) launch per vocabulary chunk (two dZ buffers)"
    return "dZ(c) launch, then one merged dW(c) + dX(c) launch per vocabulary chunk"


def workload_config(spec):
    cfg = {"workload": spec.name, "N": spec.N, "H": spec.H, "V": spec.V,
           "inputs": f"X {spec.dtype} N(0,{spec.x_std}^2)"
                     + (" RMS-normed rows" if spec.x_rms_rows else "")
                     + f", W {spec.dtype} N(0,{spec.w_std}^2)"
                     + (f" with {spec.n_scaled_w_rows} rows x{spec.w_row_scale:g}"
                        if spec.n_scaled_w_rows else "")
                     + f", labels {spec.labels}",
           "ignored_tokens": spec.n_ignore, "ignore_index": spec.ignore_index,
           "smoothing": spec.smoothing, "reduction": spec.reduction}
    return cfg


def line_config(spec, args, world: int):
    """The JSON line's `config`: the workload alone, the same on both arms
    (how our engine runs it goes under `engine`)."""
    elem = 2 if spec.dtype == "bf16" else 4
    cfg = workload_config(spec)
    cfg["l2"] = "inputs larger than L2 (W alone is %.2f GB)" % (spec.V * spec.H * elem / 1e9)
    cfg["parallelism"] = f"replicas x{world} (each rank its own batch, no collective)"
    if args.z_loss:
        cfg["z_loss"] = args.z_loss
    return cfg


# ----------------------------------------------------------------------------
# Our arm
# ----------------------------------------------------------------------------
def run_ours(args, rank: int, world: int, local_rank: int):
    import numpy as np
    import torch
    import torch.distributed as dist

    from linear_cross_entropy_logit_gb300 import build as libbuild
    from linear_cross_entropy_logit_gb300 import inputs as I

    if rank == 0:
        libbuild.build()
    if world > 1:
        dist.barrier()
    from linear_cross_entropy_logit_gb300 import binding as B

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    spec = workload_spec(args)
    wl = I.make_workload(spec, seed=args.seed + rank)
    N, H, V = spec.N, spec.H, spec.V
    B.flce_set_vocab_chunk(args.vocab_chunk)
    B.flce_set_l2_hints(args.l2_hints)
    B.flce_set_cta_pair(not args.single_cta)
    if args.multicast is not None:
        B.flce_set_cluster_multicast(bool(args.multicast))
    if args.merge is not None:
        B.flce_set_backward_merge(args.merge)
    merge_mode = B.flce_backward_merge()
    chunk = B.flce_vocab_chunk(N, H, V)

    def host_tensor(a):
        if spec.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a))

    Xh, Wh = host_tensor(wl.x), host_tensor(wl.w)
    yh = torch.from_numpy(wl.labels)
    X, W, y = Xh.to(dev), Wh.to(dev), yh.to(dev)
    dt = B.FLCE_BF16 if spec.dtype == "bf16" else B.FLCE_FP32
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    nv = torch.empty(1, dtype=torch.int32, device=dev)
    dX = torch.empty_like(X)
    dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    base_mem = torch.cuda.memory_allocated(dev)  # inputs and outputs only
    ws = B.workspace(N, H, V, dt, B.MODE_FWD_BWD, dev)

    mc_launches = [0]  # GEMM launches that took the operand-multicast walk
    if args.vocab_shards > 1:
        P = args.vocab_shards
        bounds = [round(V * i / P / 256) * 256 for i in range(P)] + [V]
        opt = B.make_options(spec.ignore_index, spec.smoothing, spec.reduction, args.z_loss)
        max_vs = max(b1 - b0 for b0, b1 in zip(bounds, bounds[1:]))
        ws = B.workspace(N, H, max_vs, dt, B.MODE_FWD_BWD, dev)
        parts = torch.empty(P, N, 4, dtype=torch.float32, device=dev)
        dxp = [torch.empty(N, H, dtype=torch.float32, device=dev) for _ in range(P)]
        dXf = torch.empty(N, H, dtype=torch.float32, device=dev)

        def step():
            n = 0
            for i, (b0, b1) in enumerate(zip(bounds, bounds[1:])):
                B.flce_forward_vocab_shard(X, W[b0:b1], y, b0, V, opt, partials=parts[i],
                                           workspace_buf=ws, err_word=err, stream=stream)
                n += B.last_launch_count()
            B.flce_combine_vocab_shards(parts, y, V, opt, loss=loss, lse=lse, valid_count=nv,
                                        err_word=err, stream=stream)
            n += B.last_launch_count()
            for i, (b0, b1) in enumerate(zip(bounds, bounds[1:])):
                B.flce_backward_vocab_shard(X, W[b0:b1], y, b0, V, lse, nv, opt,
                                            dX_partial=dxp[i], dW_shard=dW[b0:b1],
                                            workspace_buf=ws, err_word=err, stream=stream)
                n += B.last_launch_count()
            torch.sum(torch.stack(dxp), dim=0, out=dXf)  # stands in for the all-reduce
            return n
    else:
        def step():
            B.flce_fwd_bwd(X, W, y, spec.ignore_index, spec.smoothing, spec.reduction, loss=loss,
                           lse=lse, valid_count=nv, dX=dX, dW=dW, workspace_buf=ws, err_word=err,
                           stream=stream, z_loss=args.z_loss,
                           skip_ignored_blocks=args.skip_ignored, grad_filter=args.grad_filter)
            mc_launches[0] += B.last_multicast_launches()
            return B.last_launch_count()
    if args.vocab_shards > 1:
        args.no_e2e = True  # the end-to-end leg times the unsharded call only

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} after warm-up")

    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[local_rank] \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else str(local_rank)
    B.flce_profile_reset()
    B.flce_profile_enable(True)
    sampler = ClockSampler(gpu_index, args.clocks_dir) if rank == 0 else None
    time.sleep(0.2 if sampler else 0.0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    ev0.record(stream)
    launches = 0
    mc_launches[0] = 0
    for _ in range(args.steps):
        launches += step()
    launches_mc = mc_launches[0]
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    peak_extra = torch.cuda.max_memory_allocated(dev) - base_mem
    B.flce_profile_enable(False)
    prof = B.flce_profile_read()
    ms = ev0.elapsed_time(ev1)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} in the timed region")
    ms_per_step = ms / args.steps
    tokens_per_s = world * N * args.steps / (ms / 1e3)

    # --- end-to-end through the C ABI with host buffers --------------------
    # Every step copies its inputs (X, W, labels) from pinned host memory and
    # reads its result back: the loss (the `e2e` key), or with read_all every
    # output, loss, lse, dX and dW (the `e2e_all_outputs` key).  Device buffers
    # are double-buffered so that step k+1's upload and step k-1's download
    # overlap step k's fused call (three streams ordered by events); the timed
    # region runs from the first upload to the last download.
    e2e = e2e_all = None
    if not args.no_e2e:
        Xp, Wp, yp = Xh.pin_memory(), Wh.pin_memory(), yh.pin_memory()
        h2d = Xp.numel() * Xp.element_size() + Wp.numel() * Wp.element_size() + yp.numel() * 8
        ncs = max(1, args.copy_streams)
        ups = [torch.cuda.Stream(dev) for _ in range(ncs)]
        downs = [torch.cuda.Stream(dev) for _ in range(ncs)]
        s_up, s_down = ups[0], downs[0]

        def split_copy(dsts, srcs, streams, wait_ev, done_ev):
            """dst.copy_(src) for each pair, large tensors cut in row pieces spread
            over the streams; done_ev (on streams[0]) fires when all are done."""
            pieces = []
            for d, s_ in zip(dsts, srcs):
                n = d.shape[0] if d.dim() else 1
                cut = min(len(streams), n) if d.numel() * d.element_size() > (64 << 20) else 1
                step_rows = (n + cut - 1) // cut
                for i in range(cut):
                    pieces.append((d[i * step_rows:(i + 1) * step_rows],
                                   s_[i * step_rows:(i + 1) * step_rows]) if cut > 1 else (d, s_))
            for j, (d, s_) in enumerate(pieces):
                st = streams[j % len(streams)]
                with torch.cuda.stream(st):
                    st.wait_event(wait_ev)
                    d.copy_(s_, non_blocking=True)
            for st in streams[1:]:
                e = torch.cuda.Event()
                e.record(st)
                streams[0].wait_event(e)
            done_ev.record(streams[0])

        def e2e_loop(read_all):
            slots = []
            for b in range(2):
                if b == 0:
                    dev_in = (X, W, y)
                    dev_out = (loss, lse, dX, dW)
                else:
                    dev_in = (torch.empty_like(X), torch.empty_like(W), torch.empty_like(y))
                    dev_out = (torch.empty_like(loss), torch.empty_like(lse),
                               torch.empty_like(dX), torch.empty_like(dW))
                read = dev_out if read_all else dev_out[:1]
                host_out = tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in read)
                slots.append({"in": dev_in, "out": dev_out, "read": read, "host": host_out,
                              "nv": torch.empty_like(nv),
                              "ev_in": torch.cuda.Event(), "ev_comp": torch.cuda.Event(),
                              "ev_out": torch.cuda.Event()})
            d2h = sum(t.numel() * t.element_size() for t in slots[0]["read"])

            def e2e_step(k):
                sl = slots[k % 2]
                xd, wd, yd = sl["in"]
                # step k-2 no longer reads these inputs once its fused call is done
                split_copy((xd, wd, yd), (Xp, Wp, yp), ups, sl["ev_comp"], sl["ev_in"])
                stream.wait_event(sl["ev_in"])
                stream.wait_event(sl["ev_out"])         # step k-2's results are downloaded
                lo, ls, dx, dw = sl["out"]
                B.flce_fwd_bwd(xd, wd, yd, spec.ignore_index, spec.smoothing, spec.reduction,
                               loss=lo, lse=ls, valid_count=sl["nv"], dX=dx, dW=dw,
                               workspace_buf=ws, err_word=err, stream=stream,
                               z_loss=args.z_loss, skip_ignored_blocks=args.skip_ignored,
                               grad_filter=args.grad_filter)
                sl["ev_comp"].record(stream)
                split_copy(sl["host"], sl["read"], downs, sl["ev_comp"], sl["ev_out"])

            for k in range(max(args.warmup, 2)):
                e2e_step(k)
            torch.cuda.synchronize(dev)
            if world > 1:
                dist.barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_up)
            for k in range(args.steps):
                e2e_step(k)
            e1.record(s_down)
            torch.cuda.synchronize(dev)
            ems = e0.elapsed_time(e1)
            if world > 1:
                t = torch.tensor([ems], device=dev)
                dist.all_reduce(t, op=dist.ReduceOp.MAX)
                ems = float(t.item())
            if int(err.item()) != 0:
                raise RuntimeError(f"device error word {int(err.item())} in the end-to-end loop")
            host_loss = float(slots[(args.steps - 1) % 2]["host"][0].item())
            return {"value": world * N * args.steps / (ems / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "ms_per_step": ems / args.steps, "loss_read_back": host_loss,
                    "read_back": "loss, lse, dX, dW" if read_all else "loss",
                    "overlap": "uploads and downloads of neighbouring steps overlap the fused "
                               "call",
                    "copy_streams_per_direction": ncs}

        e2e = e2e_loop(False)
        e2e_all = e2e_loop(True)

    if rank != 0:
        return

    pk = peaks()
    flops_step = 8.0 * N * V * H
    skip_info = None
    if args.skip_ignored:
        rows = 128 if args.single_cta else 256
        nblk = (N + rows - 1) // rows
        lab = np.full(nblk * rows, spec.ignore_index, dtype=np.int64)
        lab[:N] = wl.labels
        active = np.any(lab.reshape(nblk, rows) != spec.ignore_index, axis=1)
        frac = float(np.minimum(rows, N - np.arange(nblk) * rows)[active].sum()) / N
        skip_info = {"block_rows": rows, "active_token_fraction": frac,
                     "note": "value counts all N tokens; tflops counts 8NVH over all N tokens "
                             "(dense-equivalent); tflops_executed counts only active blocks"}
    tflops = flops_step / (ms_per_step / 1e3) / 1e12
    # algorithmic bytes of one step: X, W read; dX, dW written; labels, lse
    elem = 2 if spec.dtype == "bf16" else 4
    bytes_step = N * H * elem * 2 + V * H * elem + V * H * 4 + N * 8 + N * 4
    # Peaks: the stated one follows the length of the timed loop (see
    # peak_choice); the fractions of both measured figures are printed.
    pname, pval, pwhy = peak_choice(pk, wall)
    t_hbm = bytes_step / (pk["hbm_gbs"] * 1e9)
    t_tensor = flops_step / (pval * 1e12)
    step_frac = max(t_tensor, t_hbm) / (ms_per_step / 1e3)
    step_frac_burst = max(flops_step / (pk["bf16_burst"] * 1e12), t_hbm) / (ms_per_step / 1e3)
    step_frac_sus = max(flops_step / (pk["bf16_sustained"] * 1e12), t_hbm) / (ms_per_step / 1e3)

    # dominant kernel: largest share of the profiled device time
    kinds = {}
    flops_kind = kind_flops(B, N, H, V, args,
                            merged=merge_mode if prof["bwd_merged"][1] > 0 else 0)
    total_prof_ms = sum(v[0] for v in prof.values()) or 1.0
    for name, (kms, n) in prof.items():
        if n == 0:
            continue
        kinds[name] = {"launches": n, "ms_total": kms, "ms_per_launch": kms / n,
                       "share_of_gemm_time": kms / total_prof_ms,
                       "flops_per_step": flops_kind[name],
                       "tflops": flops_kind[name] * args.steps / (kms / 1e3) / 1e12}
    dom = max(kinds, key=lambda k: kinds[k]["ms_total"]) if kinds else None
    roofline = None
    dense_default = not (args.skip_ignored or args.grad_filter or args.vocab_shards > 1 or
                         args.shape or args.single_cta or args.l2_hints or
                         args.merge is not None or args.vocab_chunk or
                         args.multicast is not None)
    traffic = load_traffic(spec.name) if dense_default else None
    if dom:
        ach = kinds[dom]["tflops"]
        src = "measured (MEASURED_PEAKS.json)" if pk["source"] == "measured" else "fallback"
        roofline = {"bound": "tensor", "achieved": ach, "peak": pval,
                    "unit": "TFLOP/s", "frac": ach / pval,
                    "traffic": traffic.get(dom) if traffic else None,
                    "kernel": dom,
                    "peak_source": f"{src} bf16 {pname}: the kernel is timed per launch "
                                   f"({kinds[dom]['ms_per_launch']:.3f} ms) inside a "
                                   f"{wall:.2f} s loop of back-to-back steps; {pwhy}",
                    "peak_burst": pk["bf16_burst"],
                    "frac_of_burst": ach / pk["bf16_burst"],
                    "peak_sustained": pk["bf16_sustained"],
                    "frac_of_sustained": ach / pk["bf16_sustained"]}

    cpu = None
    if args.cpu_baseline_rows > 0 and world == 1:
        r, secs = oracle_sample(wl, args.cpu_baseline_rows, args.z_loss)
        cpu = {"value": r / secs, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"first {r} of {N} tokens, full V={V} and H={H}, fp64 oracle "
                         f"forward+backward (numpy float64 matmul), {secs:.1f} s"}

    extra = {"workspace_bytes": ws.numel(),
             "workspace_vs_nxv_bf16": ws.numel() / (N * V * 2),
             "dz_chunk_bytes": N * chunk * 2,
             "dz_buffers": 2 if (merge_mode == 1 and B.flce_cta_pair()) else 1,
             "peak_extra_device_bytes": peak_extra,
             "nxv_bf16_bytes": N * V * 2}
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": spec.dtype, "data": "synthetic",
        "config": line_config(spec, args, world),
        "engine": {"vocab_chunk": chunk,
                   "tiles": "128x256 single CTA" if args.single_cta else "256x256 CTA pair",
                   "cluster_multicast": (not args.single_cta) and B.flce_cluster_multicast(),
                   "backward": backward_layout(merge_mode, args),
                   "skip_ignored_blocks": args.skip_ignored,
                   "grad_filter": args.grad_filter or None,
                   "vocab_shards": args.vocab_shards or None,
                   "l2_hints": args.l2_hints},
        "tflops": tflops,
        "skip": skip_info,
        "tflops_executed": tflops * skip_info["active_token_fraction"] if skip_info else tflops,
        "step_roofline": {"bound": "tensor" if t_tensor >= t_hbm else "hbm",
                          "frac": step_frac, "flops": flops_step, "bytes": bytes_step,
                          "peak_tflops": pval,
                          "peak_source": f"{pk['source']} bf16 {pname}",
                          "frac_of_burst": step_frac_burst,
                          "peak_tflops_burst": pk["bf16_burst"],
                          "frac_of_sustained": step_frac_sus,
                          "peak_tflops_sustained": pk["bf16_sustained"]},
        "roofline": roofline,
        "kernels": kinds,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "e2e_all_outputs": e2e_all,
        "gpu_launches": launches,
        "gpu_launches_multicast": launches_mc,
        "clocks": clocks,
        "wall_s_timed": wall,
        "memory": extra,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.summarize_traffic:
        shape = tuple(int(v) for v in args.shape.split(",")) if args.shape else None
        summarize_traffic(args.summarize_traffic, args.workload, shape)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    import torch.distributed as dist
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
