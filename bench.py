"""Benchmark of the PISA prefill hot path (pyramid + block selection + sparse attention).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pisa|reference] [--workload NAME]

One step = one pass of the whole hot path over one batch of synthetic input: build the
key pyramid, select blocks for every query (level walk, exact leaf LSE, top-K) and attend
over the selected blocks.  The default workload is the selection-scale prefill
(N = 262144 tokens, H_q = 16, H_kv = 1, d = 128, C = 64, g = 2, K = 16); its inputs (1.2 GB)
are resident in HBM and larger than the 129 MB L2, so no flush is needed between steps.

Under torchrun every rank runs its own replica on its own GPU (the path has no exchange
step: weak scaling); the timed region is bracketed by a barrier and a synchronize, and
rank 0 prints one JSON line with the maximum time over ranks.

--impl reference times the CPU oracle (the plain statement of the method used by the
tests) on a bounded sample of the same workload; only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill tokens/s (select + sparse attn)"
UNIT = "tokens/s"
KERNELS_PER_STEP = 10  # pyramid 2, stage 1 (with the clustering histogram), clustering 4 (three scans, scatter and tiles in one), leaf LSE, top-K, attention

# The paper's own figures for this path (summary page "Block Sparse Attention with Log-Linear
# Complexity", section "Experimental results", item 5, Fig. 3): context only.  They are ratios
# against the authors' BSA selection on hardware the page does not name; no absolute latency,
# throughput or decode time is given there.
PAGES_REFERENCE = {
    "selection_speedup_vs_bsa": {"64K": 2.86, "128K": 5.31, "256K": 9.95},
    "setting": "block selection at C=64, K=8 (this bench times K=8 under secondary.prefill_*_k8)",
    "hardware": "not stated on the page",
    "note": "BSA is faster than PISA at 4K-16K on the page's figure",
}

# DRAM traffic of the attention kernel per launch on the 256K prefill (dram__bytes_read.sum +
# dram__bytes_write.sum from one ncu capture; the committed DRAM-traffic profile of that
# workload), keyed by a hash of the kernel's sources: when the sources change the figure is
# stale and is reported as null until it is taken again.
ATTN_TRAFFIC = {"sources_sha256": "9ed724c54f00616b0cb692bf96f4336023006022014a0b1f66ec429cbc54faf3",
                "workload": "prefill_256k", "bytes": 14359143936 + 1091798784}
ATTN_SOURCES = ["hierarchical_top_block_gb300/csrc/sparse_attn.cu", "hierarchical_top_block_gb300/csrc/common.cuh",
                "hierarchical_top_block_gb300/csrc/kernels.cuh"]


def attn_sources_sha256():
    import hashlib

    h = hashlib.sha256()
    for rel in ATTN_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="pisa", choices=["pisa", "reference"])
    ap.add_argument("--workload", default="prefill_256k")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--no-secondary", action="store_true", help="skip the 32K prefill and decode measurements")
    ap.add_argument("--cpu-sample-rows", type=int, default=32768)
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg (profiling runs)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline (profiling runs)")
    ap.add_argument("--profile-section", choices=["decode", "bsa"], default=None,
                    help="run only the decode step or the PISA/BSA selection timing, at a reduced size, and print "
                         "its JSON (for profiler captures; --steps and --warmup apply)")
    ap.add_argument("--profile-batch", type=int, default=8, help="decode batch of --profile-section decode")
    ap.add_argument("--profile-n", type=int, default=65536, help="sequence length of --profile-section bsa")
    return ap.parse_args()


# ------------------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ------------------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def init_dist(backend):
    import torch.distributed as dist

    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of the ranks' values (every rank gets it)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names[1:], parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------
# algorithmic work of the attention step (counted from the realised selection)
# ------------------------------------------------------------------------------------
def attention_work(idx, N, H_q, H_kv, d, C=64):
    """Algorithmic work of one attention launch, counted from the realised selection.

    flops: 4 d per visible (query head, key) pair of the selected blocks (QK^T and PV).
    gather_bytes: the K and V rows of every selected, visible block, once per (query, KV head)
    group (C keys x d x 2 bytes x 2 tensors per block): what the kernel reads from L2.
    """
    import torch

    t = torch.arange(N, device=idx.device, dtype=torch.int64).view(1, 1, N, 1)
    j = idx.to(torch.int64)
    vis = torch.clamp(t - j * C + 1, min=0, max=C) * (j >= 0)
    keys_per_group_query = vis.sum().item()  # over (b, h_kv, t)
    blocks = (vis > 0).sum().item()
    return {"flops": 4.0 * d * keys_per_group_query * (H_q // H_kv), "gather_bytes": blocks * C * d * 2 * 2,
            "blocks": blocks}


def level_sizes(n, C=64, g=2):
    """Nodes per pyramid level for n tokens: M_1 = ceil(n / C), M_{l+1} = ceil(M_l / g)."""
    out = [-(-n // C)] if n > 0 else []
    while out and out[-1] > 1:
        out.append(-(-out[-1] // g))
    return out


def stage1_work(N, H_q, H_kv, d, K, B=1, C=64, causal=True):
    """Child rows the level walk scores, summed over the queries, for a walk whose survivors
    always have all their children (an upper bound of the realised walk, exact away from the
    causal edge): at level l the candidates are min(eligible, 2 x survivors of level l + 1);
    a level is scored when more than K remain, each candidate by its 2 children."""
    import numpy as np

    M = level_sizes(N, C)
    L = len(M)
    t = np.arange(N, dtype=np.int64)
    surv = np.ones(N, dtype=np.int64)  # the root
    rows = np.zeros(N, dtype=np.int64)
    for lvl in range(L - 1, 1, -1):       # levels L-1 .. 2 (1-based); M[lvl - 1] nodes
        span = C << (lvl - 1)             # keys covered by one level-lvl node
        elig = np.minimum(M[lvl - 1], t // span + 1) if causal else np.full(N, M[lvl - 1])
        cand = np.minimum(elig, 2 * surv)
        scored = cand > K
        rows += np.where(scored, 2 * cand, 0)
        surv = np.minimum(cand, K)
    G = H_q // H_kv
    total_rows = int(rows.sum()) * B * H_kv
    return {"child_rows": total_rows, "flops": 2.0 * d * G * total_rows, "l2_gather_bytes": total_rows * d * 2}


def leaf_lse_work(s2, N, H_q, H_kv, d, C=64):
    """Algorithmic work of Stage 2, counted from the realised level-2 survivors s2
    [B, H_kv, N, K]: 2 d flops per (query head, visible key) of each eligible leaf child."""
    import torch

    t = torch.arange(N, device=s2.device, dtype=torch.int64).view(1, 1, N, 1)
    node = s2.to(torch.int64)
    keys = 0
    for c in (0, 1):
        leaf = 2 * node + c
        vis = torch.clamp(torch.minimum(t, torch.tensor(N - 1, device=s2.device)) - leaf * C + 1, min=0, max=C)
        keys += int((vis * (node >= 0)).sum().item())
    return {"visible_keys": keys, "flops": 2.0 * d * keys * (H_q // H_kv)}


def roofline_entry(kernel, ms, bound, work, pk):
    """One kernel's roofline: algorithmic work per launch / its event-timed duration, against the
    measured peak (HBM copy bandwidth, or bf16 dense burst)."""
    if bound == "hbm":
        ach = work / (ms * 1e-3) / 1e9
        return {"kernel": kernel, "bound": "hbm", "ms": ms, "algorithmic_bytes": work, "achieved": ach,
                "peak": pk["hbm"], "unit": "GB/s", "frac": ach / pk["hbm"], "peak_source": pk["source"] + " copy"}
    ach = work / (ms * 1e-3) / 1e12
    return {"kernel": kernel, "bound": "tensor", "ms": ms, "algorithmic_flops": work, "achieved": ach,
            "peak": pk["tensor"], "unit": "TFLOP/s", "frac": ach / pk["tensor"],
            "peak_source": pk["source"] + " bf16 dense burst"}


def phase_rooflines(w, step_fn, s2, attn_flops, steps=5):
    """Runs `steps` more steps with the library's per-phase event timing on and returns a
    roofline entry per kernel of the step (CUDA events recorded by the library on the
    launching stream around each kernel phase)."""
    import torch

    import hierarchical_top_block_gb300 as pisa

    pisa.pisa_phase_timing(True)
    for _ in range(steps):
        step_fn()
    torch.cuda.synchronize()
    times = pisa.pisa_phase_times()
    pisa.pisa_phase_timing(False)
    ms = {k: v[0] / v[1] for k, v in times.items() if v[1] > 0}
    pk = peaks()
    B, N, H_q, H_kv, d, K = w.B, w.N, w.H_q, w.H_kv, w.d, w.K
    nodes = sum(level_sizes(N))
    q_bytes = B * N * H_q * d * 2
    kv_bytes = B * H_kv * N * d * 2
    sel_int = B * H_kv * N * K * 4
    s1 = stage1_work(N, H_q, H_kv, d, K, B)
    s2w = leaf_lse_work(s2, N, H_q, H_kv, d)
    out = {}
    if "pyramid" in ms:
        out["pyramid"] = roofline_entry("pyramid_leaves_kernel + pyramid_upper_kernel", ms["pyramid"], "hbm",
                                        kv_bytes + B * H_kv * nodes * d * 2, pk)
    if "stage1" in ms:
        e = roofline_entry("stage1_kernel", ms["stage1"], "hbm", q_bytes + 2 * sel_int, pk)
        e["mma_flops"] = s1["flops"]
        e["mma_tflops"] = s1["flops"] / (ms["stage1"] * 1e-3) / 1e12
        e["l2_gather_bytes"] = s1["l2_gather_bytes"]
        e["note"] = "HBM bytes: Q once, survivors and list places out; mma_flops: saturated-walk count"
        out["stage1"] = e
    if "cluster" in ms:
        out["cluster"] = roofline_entry("cluster kernels (5)", ms["cluster"], "hbm", 3 * sel_int, pk)
    if "leaf_lse" in ms:
        e = roofline_entry("leaf_lse_kernel", ms["leaf_lse"], "tensor", s2w["flops"], pk)
        e["visible_keys"] = s2w["visible_keys"]
        out["leaf_lse"] = e
    if "topk" in ms:
        out["topk"] = roofline_entry("topk_kernel", ms["topk"], "hbm", sel_int + 2 * sel_int + sel_int, pk)
    if "sparse_attn" in ms:
        out["sparse_attn"] = roofline_entry("sparse_attn_kernel", ms["sparse_attn"], "tensor", attn_flops, pk)
    out["timed_steps"] = steps
    out["method"] = ("CUDA events the library records on the launching stream around each kernel phase "
                     "(pisa_phase_timing), over separate steps after the timed region")
    return out


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=p["hbm_gbs"], tensor=p["bf16_tflops"], tensor_sustained=p.get("bf16_tflops_sustained"),
                    source="measured")
    return dict(hbm=6800.0, tensor=1900.0, tensor_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------------------------
# the GPU path
# ------------------------------------------------------------------------------------
def run_pisa(args):
    import torch

    import hierarchical_top_block_gb300 as pisa
    import workloads as W

    from hierarchical_top_block_gb300.build import build

    build()  # no-op when the library is current
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    backend = "nccl" if world > 1 else "gloo"
    init_dist(backend)
    dev = torch.device("cuda", local)
    w = W.WORKLOADS[args.workload]
    assert w.decode_steps == 0, "the timed step is a prefill workload"

    Q, K, V = W.prefill_inputs(w, dev)
    P = torch.empty(w.B, w.H_kv, pisa.pisa_pyramid_nodes(w.N), w.d, dtype=torch.bfloat16, device=dev)
    shape = pisa.make_shape(w.B, w.N, w.H_q, w.H_kv, w.d)
    params = pisa.make_params(w.K)
    ws = torch.empty(pisa.pisa_select_workspace_bytes(shape, params), dtype=torch.uint8, device=dev)
    idx = torch.empty(w.B, w.H_kv, w.N, w.K, dtype=torch.int32, device=dev)
    O = torch.empty_like(Q)
    LSE = torch.empty(w.B, w.H_q, w.N, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    s2 = torch.empty(w.B, w.H_kv, w.N, w.K, dtype=torch.int32, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step(marks=None, keep_s2=False):
        if marks is not None:
            marks[0].record(stream)
        pisa.pisa_build_pyramid(K, P=P)
        pisa.pisa_select_prefill(Q, K, P, w.K, ws=ws, idx=idx, s2=s2 if keep_s2 else None)
        if marks is not None:
            marks[1].record(stream)
        pisa.pisa_sparse_attn_prefill(Q, K, V, idx, O=O, LSE=LSE)
        if marks is not None:
            marks[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if pisa.pisa_get_last_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")
    marks = [[ev(), ev(), ev()] for _ in range(args.steps)]
    clocks = ClockSampler(dev.index)
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = ev(), ev()
    t0.record(stream)
    for i in range(args.steps):
        step(marks[i])
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    err = pisa.pisa_get_last_device_error()
    if err != 0:
        raise RuntimeError(f"device error word {err} during the timed region")
    ms_local = t0.elapsed_time(t1) / args.steps
    ms = max_over_ranks(ms_local, world, dev if backend == "nccl" else None)
    sel_ms = statistics.mean(m[0].elapsed_time(m[1]) for m in marks)
    att_ms = statistics.mean(m[1].elapsed_time(m[2]) for m in marks)
    tokens = w.B * w.N
    value = tokens * world / (ms * 1e-3)

    work = attention_work(idx, w.N, w.H_q, w.H_kv, w.d)
    flops = work["flops"]
    pk = peaks()
    rooflines = section(phase_rooflines, w, lambda: step(keep_s2=True), s2, flops)
    achieved_tf = flops / (att_ms * 1e-3) / 1e12
    io_bytes = sum(x.numel() * x.element_size() for x in (Q, K, V, O, LSE, P, idx))
    traffic = ATTN_TRAFFIC["bytes"] if (ATTN_TRAFFIC["sources_sha256"] == attn_sources_sha256()
                                        and ATTN_TRAFFIC["workload"] == w.name) else None
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded counter-based generator; block-mean key offsets)",
        "config": {"workload": w.name, "B": w.B, "N": w.N, "H_q": w.H_q, "H_kv": w.H_kv, "d": w.d, "C": w.C,
                   "g": w.g, "K": w.K, "causal": True, "parallelism": f"replicas x{world}",
                   "l2": f"inputs and outputs ({io_bytes / 1e9:.2f} GB) larger than L2 (129 MB), no flush"},
        "breakdown_ms": {"pyramid+selection": sel_ms, "sparse_attention": att_ms},
        "selection_only_tokens_per_s": tokens * world / (sel_ms * 1e-3),
        "roofline": {"kernel": "sparse_attn_kernel", "bound": "tensor", "achieved": achieved_tf,
                     "peak": pk["tensor"], "unit": "TFLOP/s", "frac": achieved_tf / pk["tensor"],
                     "traffic": traffic, "algorithmic_flops_per_launch": flops,
                     "peak_source": pk["source"] + " bf16 dense burst",
                     "l2_gather": {"bytes_per_launch": work["gather_bytes"], "blocks": work["blocks"],
                                   "achieved_tbs": work["gather_bytes"] / (att_ms * 1e-3) / 1e12}},
        "rooflines": rooflines,
        "clocks": clk,
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "pages_reference": PAGES_REFERENCE,
    }
    if rank == 0 and not args.no_secondary:
        out["scoring_variants"] = section(scoring_variants, Q, K, P, w, ws, idx)
        out["backward"] = section(backward_section, Q, K, V, idx, O, LSE, w, work)
    if rank == 0:
        out["e2e"] = None if args.no_e2e else section(run_e2e, args, w, dev)
        if not args.no_secondary:
            # K = 8 is the setting of the paper's selection-speed comparison (its Fig. 3)
            out["secondary"] = {
                "prefill_32k": section(secondary_prefill, W.WORKLOADS["prefill_32k"], dev),
                "prefill_32k_k8": section(secondary_prefill, W.WORKLOADS["prefill_32k"], dev, K_sel=8),
                "prefill_256k_k8": section(secondary_prefill, W.WORKLOADS["prefill_256k"], dev, K_sel=8),
                "decode_128k": section(secondary_decode, W.WORKLOADS["decode_128k"], dev),
                "bsa_vs_pisa_selection": section(bsa_vs_pisa_section, dev),
                "selection_quality_32k": section(selection_quality_section, W.WORKLOADS["prefill_32k"], dev)}
        out["cpu_baseline"] = None if args.no_cpu else cpu_baseline(args, w)
        print(json.dumps(out), flush=True)
    barrier(world)


def section(fn, *args, **kwargs):
    """Runs one of the line's secondary sections; one that fails is reported in its place
    ({"error": ...}) instead of costing the whole line (the timed step is checked before)."""
    try:
        return fn(*args, **kwargs)
    except Exception as e:  # noqa: BLE001 - any failure of a secondary section is reported
        return {"error": f"{type(e).__name__}: {e}"}


def backward_section(Q, K, V, idx, O, LSE, w, work, steps=5, warmup=3):
    """The attention backward (dQ, dK, dV over the selected blocks) on the bench inputs with a
    seeded upstream gradient.  Algorithmic flops: per visible (query head, key) pair,
    2d each for S, dP and dQ (dQ kernel) and for S^T, dP^T, dV and dK (dK/dV kernel)."""
    import torch

    import hierarchical_top_block_gb300 as pisa

    gen = torch.Generator(device="cpu").manual_seed(99)
    dO = (torch.randn(Q.shape, generator=gen) * 0.5).to(torch.bfloat16).to(Q.device)
    B, N, H_q, d = Q.shape
    shape = pisa.make_shape(B, N, H_q, K.shape[1], d, K.shape[2])
    ws = torch.empty(pisa.pisa_attn_backward_workspace_bytes(shape, pisa.make_params(w.K)), dtype=torch.uint8,
                     device=Q.device)
    dQ = torch.empty(Q.shape, dtype=torch.float32, device=Q.device)
    dK = torch.empty(K.shape, dtype=torch.float32, device=Q.device)
    dV = torch.empty_like(dK)
    run = lambda: pisa.pisa_sparse_attn_backward(Q, K, V, idx, O, LSE, dO, ws=ws, dQ=dQ, dK=dK, dV=dV)  # noqa: E731
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        run()
    b.record()
    torch.cuda.synchronize()
    if pisa.pisa_get_last_device_error() != 0:
        raise RuntimeError("device error word set during the backward")
    ms = a.elapsed_time(b) / steps
    flops = work["flops"] / 4.0 * 14.0   # forward counts 4d per pair; the backward 14d
    del dO, ws, dQ, dK, dV
    torch.cuda.empty_cache()
    return {"ms": ms, "tokens_per_s": B * N / (ms * 1e-3), "algorithmic_tflop": flops / 1e12,
            "achieved_tflops": flops / (ms * 1e-3) / 1e12}


def scoring_variants(Q, K, P, w, ws, idx, steps=10, warmup=3):
    """Selection-only time (pyramid + selection) on the same inputs for the three block
    scorings: the LSE (PISA) and its first- and second-order truncations (PISA-1, PISA-2)."""
    import torch

    import hierarchical_top_block_gb300 as pisa

    res = {}
    for name in ("lse", "pisa1", "pisa2"):
        def sel():
            pisa.pisa_build_pyramid(K, P=P)
            pisa.pisa_select_prefill(Q, K, P, w.K, ws=ws, idx=idx, scoring=name)
        for _ in range(warmup):
            sel()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            sel()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        res[name] = {"select_ms": ms, "selection_tokens_per_s": w.B * w.N / (ms * 1e-3)}
    if pisa.pisa_get_last_device_error() != 0:
        raise RuntimeError("device error word set while timing the scoring variants")
    return res


def run_e2e(args, w, dev):
    """Same metric through the host-buffer entry point: H2D of Q, K, V and D2H of O and LSE
    inside the timed region, every step."""
    import torch

    import hierarchical_top_block_gb300 as pisa
    import workloads as W

    Qh = W.make_q(w, dev).cpu().pin_memory()
    Kh = W.make_kv(w, "K", dev).cpu().pin_memory()
    Vh = W.make_kv(w, "V", dev).cpu().pin_memory()
    Oh = torch.empty_like(Qh).pin_memory()
    Lh = torch.empty(w.B, w.H_q, w.N, dtype=torch.float32).pin_memory()
    shape = pisa.make_shape(w.B, w.N, w.H_q, w.H_kv, w.d)
    params = pisa.make_params(w.K)
    dws = torch.empty(pisa.pisa_prefill_host_workspace_bytes(shape, params), dtype=torch.uint8, device=dev)
    pisa.pisa_prefill_host(Qh, Kh, Vh, w.K, dev_ws=dws, O_host=Oh, LSE_host=Lh, device=dev.index)
    torch.cuda.synchronize()
    calls = []
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        tc = time.perf_counter()
        pisa.pisa_prefill_host(Qh, Kh, Vh, w.K, dev_ws=dws, O_host=Oh, LSE_host=Lh, device=dev.index)
        calls.append(round((time.perf_counter() - tc) * 1e3, 3))  # each call returns when all its work is done
    dt = (time.perf_counter() - t0) / args.e2e_steps
    h2d = Qh.numel() * 2 + Kh.numel() * 2 + Vh.numel() * 2
    d2h = Oh.numel() * 2 + Lh.numel() * 4
    return {"value": w.B * w.N / dt, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": dt * 1e3, "steps": args.e2e_steps, "calls_ms": calls,
            "api": "pisa_prefill_host (pinned host buffers)"}


def secondary_prefill(w, dev, steps=5, K_sel=None):
    """Pyramid + selection + attention, and pyramid + selection alone, on a workload's inputs
    (K_sel overrides the workload's K)."""
    import torch

    import hierarchical_top_block_gb300 as pisa
    import workloads as W

    Ks = w.K if K_sel is None else K_sel
    Q, K, V = W.prefill_inputs(w, dev)
    P = pisa.pisa_build_pyramid(K)
    shape = pisa.make_shape(w.B, w.N, w.H_q, w.H_kv, w.d)
    ws = torch.empty(pisa.pisa_select_workspace_bytes(shape, pisa.make_params(Ks)), dtype=torch.uint8, device=dev)
    idx = torch.empty(w.B, w.H_kv, w.N, Ks, dtype=torch.int32, device=dev)
    O = torch.empty_like(Q)
    L = torch.empty(w.B, w.H_q, w.N, dtype=torch.float32, device=dev)

    def select():
        pisa.pisa_build_pyramid(K, P=P)
        pisa.pisa_select_prefill(Q, K, P, Ks, ws=ws, idx=idx)

    def step():
        select()
        pisa.pisa_sparse_attn_prefill(Q, K, V, idx, O=O, LSE=L)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    ms, sel_ms = timed(step), timed(select)
    if pisa.pisa_get_last_device_error() != 0:
        raise RuntimeError("device error word set during the secondary prefill")
    return {"tokens_per_s": w.B * w.N / (ms * 1e-3), "ms_per_step": ms,
            "selection_tokens_per_s": w.B * w.N / (sel_ms * 1e-3), "select_ms": sel_ms,
            "N": w.N, "H_q": w.H_q, "H_kv": w.H_kv, "K": Ks}


def bsa_vs_pisa_section(dev, Ns=(4096, 16384, 65536, 131072, 262144), K_sel=8, steps=10):
    """Block-selection latency of PISA (pyramid + pisa_select_prefill) and of the BSA flat
    selection (pyramid + pisa_select_bsa) at the pages' Fig. 3 setting (C = 64, K = 8) on the
    selection-scale shape (H_q = 16, H_kv = 1, d = 128), for N from 4K to 256K; the ratio
    BSA / PISA is the speed-up the pages report (2.86x, 5.31x, 9.95x at 64K, 128K, 256K)."""
    import torch

    import hierarchical_top_block_gb300 as pisa
    import workloads as W

    base = W.WORKLOADS["prefill_256k"]
    rows = []
    for N in Ns:
        w = base.with_(N=N)
        Q, K, V = W.prefill_inputs(w, dev)
        del V
        P = pisa.pisa_build_pyramid(K)
        shape = pisa.make_shape(w.B, N, w.H_q, w.H_kv, w.d)
        ws = torch.empty(pisa.pisa_select_workspace_bytes(shape, pisa.make_params(K_sel)), dtype=torch.uint8, device=dev)
        wb = torch.empty(pisa.pisa_select_bsa_workspace_bytes(shape, pisa.make_params(K_sel)), dtype=torch.uint8,
                         device=dev)
        idx = torch.empty(w.B, w.H_kv, N, K_sel, dtype=torch.int32, device=dev)

        def timed(fn):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(steps):
                fn()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / steps

        pyr = timed(lambda: pisa.pisa_build_pyramid(K, P=P))
        pisa_ms = timed(lambda: (pisa.pisa_build_pyramid(K, P=P), pisa.pisa_select_prefill(Q, K, P, K_sel, ws=ws, idx=idx)))
        bsa_ms = timed(lambda: (pisa.pisa_build_pyramid(K, P=P), pisa.pisa_select_bsa(Q, P, K_sel, ws=wb, idx=idx)))
        if pisa.pisa_get_last_device_error() != 0:
            raise RuntimeError("device error word set while timing the selections")
        rows.append({"N": N, "pyramid_ms": pyr, "pisa_select_ms": pisa_ms, "bsa_select_ms": bsa_ms,
                     "pisa_speedup_over_bsa": bsa_ms / pisa_ms})
        del Q, K, P, ws, wb, idx
        torch.cuda.empty_cache()
    return {"K": K_sel, "C": 64, "H_q": base.H_q, "H_kv": base.H_kv, "d": base.d, "rows": rows,
            "includes": "pyramid build in both selections",
            "pages_pisa_speedup_over_bsa": {"65536": 2.86, "131072": 5.31, "262144": 9.95},
            "note": ("BSA's mean-summary score is linear in q, so the group's head sum folds into one "
                     "query vector: one d-length dot product per (query, block) on the tensor cores")}


def selection_quality_section(w, dev, samples=96, seed=11):
    """Recall@K against the exact leaf-LSE top-K and kept dense-attention mass, on the seeded
    needle workload, for each block scoring and K = 8 (the pages' setting) and the workload's K;
    and the needle-hit rate: the share of the query rows each planted needle was aimed at whose
    selection holds the needle's block."""
    import numpy as np
    import torch

    import hierarchical_top_block_gb300 as pisa
    from hierarchical_top_block_gb300 import quality
    import workloads as W

    Q, K, V = W.prefill_inputs(w, dev)
    P = pisa.pisa_build_pyramid(K)
    rng = np.random.default_rng(seed)
    rows = sorted((int(rng.integers(0, w.B)), int(t)) for t in rng.integers(64, w.N, samples))
    targets = [(n.b, n.g, n.pos, t) for n in W.needles(w) for (t, _h) in n.rows]
    res = {"samples": samples, "workload": w.name, "needle_rows": len(targets),
           "reference": "exact top-K of the head-summed leaf LSE over all eligible blocks (own block kept)"}
    for K_sel in sorted({8, w.K}):
        for name in ("lse", "pisa1", "pisa2"):
            idx = pisa.pisa_select_prefill(Q, K, P, K_sel, scoring=name)
            torch.cuda.synchronize()
            rep = quality.selection_quality(Q, K, idx, K_sel, rows)
            rep["needle_hit_rate"] = quality.needle_hit_rate(idx, targets)["hit_rate"]
            res[f"K{K_sel}_{name}"] = rep
    del Q, K, V, P
    torch.cuda.empty_cache()
    return res


def secondary_decode(w, dev, steps=None, warmup=3):
    """Batched decode: per-step latency of the fused decode kernel over all 64 sequences, for
    each of the workload's decode steps (256) after a few untimed ones."""
    import torch

    import hierarchical_top_block_gb300 as pisa
    import workloads as W

    steps = w.decode_steps if steps is None else steps
    N_cap = w.N + warmup + steps
    Kc = torch.empty(w.B, w.H_kv, N_cap, w.d, dtype=torch.bfloat16, device=dev)
    Vc = torch.empty_like(Kc)
    for b in range(w.B):
        for g in range(w.H_kv):
            Kc[b, g, :w.N] = W.kv_slice(w, "K", b, g, device=dev)
            Vc[b, g, :w.N] = W.kv_slice(w, "V", b, g, device=dev)
    Pc = pisa.pisa_build_pyramid(Kc, N=w.N)
    seq = torch.full((w.B,), w.N, dtype=torch.int32, device=dev)
    ins = [W.decode_step_inputs(w, s, dev) for s in range(warmup + steps)]
    o = torch.empty(w.B, w.H_q, w.d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.B, w.H_q, dtype=torch.float32, device=dev)
    # the leaf logits scratch of pisa_decode_step_ws, allocated once
    ws = torch.empty(pisa.pisa_decode_workspace_bytes(pisa.make_shape(w.B, 0, w.H_q, w.H_kv, w.d, N_cap),
                                                      pisa.make_params(w.K)), dtype=torch.uint8, device=dev)
    for s in range(warmup):
        pisa.pisa_decode_step(*ins[s], Kc, Vc, Pc, seq, w.K, o=o, lse=lse, ws=ws)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s in range(steps):
        evs[s][0].record()
        pisa.pisa_decode_step(*ins[warmup + s], Kc, Vc, Pc, seq, w.K, o=o, lse=lse, ws=ws)
        evs[s][1].record()
    torch.cuda.synchronize()
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
    del Kc, Vc, Pc
    torch.cuda.empty_cache()
    mean_us = statistics.mean(us)
    hbm = decode_hbm_bytes(w)
    pk = peaks()
    return {"step_us_mean": mean_us, "step_us_p50": us[len(us) // 2], "steps": steps,
            "B": w.B, "cached_tokens": w.N, "H_q": w.H_q, "H_kv": w.H_kv, "note": f"{warmup} untimed steps, then {steps} timed ones",
            "roofline": {"bound": "hbm", "algorithmic_bytes_per_step": hbm,
                         "achieved": hbm / (mean_us * 1e-6) / 1e9, "peak": pk["hbm"], "unit": "GB/s",
                         "frac": hbm / (mean_us * 1e-6) / 1e9 / pk["hbm"], "peak_source": pk["source"] + " copy"}}


def decode_hbm_bytes(w, C=64, g=2):
    """Bytes one decode step must read at least, per (sequence, KV head): the child summaries
    of every scored level (2K candidates x 2 children), the raw keys of the 2K leaf candidates
    (the selected blocks' keys are among them and are not counted again), and the raw values of
    the K selected blocks; d bf16 values per row."""
    n = w.N + 1
    sizes = level_sizes(n, C, g)
    scored = sum(1 for m in sizes[1:-1] if m > w.K)  # levels 2.. whose candidates exceed K
    rows = scored * 2 * w.K * g + 2 * w.K * C + w.K * C
    return w.B * w.H_kv * rows * w.d * 2


# ------------------------------------------------------------------------------------
# the CPU oracle (baseline / reference arm)
# ------------------------------------------------------------------------------------
class OracleSample:
    """The CPU oracle on a bounded sample of the workload: the full pyramid, plus selection
    and attention for a set of query positions spread over the sequence.  Inputs are
    generated once (seeded, on the CPU); each run() is timed on its own."""

    def __init__(self, w, max_rows, seed=7):
        import numpy as np

        import oracle
        import workloads as W

        self.w = w
        self.o = oracle.Oracle()
        self.Kb = W.bits(W.make_kv(w, "K", "cpu"))
        self.Vb = W.bits(W.make_kv(w, "V", "cpu"))
        rng = np.random.default_rng(seed)
        self.ts_all = rng.permutation(w.N)[:max_rows].astype(np.int64)
        self.Qb = np.zeros((w.B, w.N, w.H_q, w.d), np.uint16)
        self.Qb[0, self.ts_all] = W.bits(W.q_rows(w, 0, self.ts_all))

    def run(self, rows_n, offset=0):
        import numpy as np

        w = self.w
        ts = np.sort(self.ts_all[offset:offset + rows_n])
        t0 = time.perf_counter()
        P = self.o.build_pyramid(self.Kb)
        rows = np.array([(0, g, t) for g in range(w.H_kv) for t in ts], np.int64).reshape(-1, 3)
        sel = self.o.select(self.Qb, self.Kb, P, w.K, rows)
        self.select_dt = time.perf_counter() - t0          # pyramid + selection alone
        idx = np.full((w.B, w.H_kv, w.N, w.K), -1, np.int32)
        idx[rows[:, 0], rows[:, 1], rows[:, 2]] = sel["idx"]
        self.o.sparse_attention(self.Qb, self.Kb, self.Vb, idx, np.stack([np.zeros_like(ts), ts], 1))
        dt = time.perf_counter() - t0
        return len(ts) / dt, dt


def cpu_baseline(args, w):
    try:
        sample = OracleSample(w, args.cpu_sample_rows)
        tps, dt = sample.run(args.cpu_sample_rows)
    except Exception as e:  # the baseline is informational
        return {"value": None, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", "error": str(e)}
    out = {"value": tps, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
           "sample": f"full pyramid + selection and attention for {args.cpu_sample_rows} query positions of "
                     f"{w.name} (N={w.N}), {dt:.1f} s wall on {os.cpu_count()} threads",
           "selection_only_tokens_per_s": args.cpu_sample_rows / sample.select_dt}
    if not args.no_secondary:
        out["secondary"] = oracle_secondary()
    return out


def oracle_secondary(rows_32k=2048, decode_steps=8):
    """The oracle on bounded samples of the other workloads, as context: the 32K prefill
    (selection alone and with attention, for a set of query positions) and the batched decode
    step (the first sequence's first two KV heads for a few steps, scaled to the whole batch
    by the number of (sequence, KV head) pairs, and labelled so)."""
    import numpy as np

    import oracle
    import workloads as W

    res = {}
    try:
        w = W.WORKLOADS["prefill_32k"]
        sample = OracleSample(w, rows_32k)
        tps, dt = sample.run(rows_32k)
        res["prefill_32k"] = {"tokens_per_s": tps, "selection_tokens_per_s": rows_32k / sample.select_dt,
                              "sample": f"full pyramid + {rows_32k} query positions, {dt:.1f} s wall"}
    except Exception as e:  # informational
        res["prefill_32k"] = {"error": str(e)}
    try:
        w = W.WORKLOADS["decode_128k"]
        o = oracle.Oracle()
        pairs = 2                                      # (sequence 0, KV heads 0 and 1)
        N_cap = w.N + decode_steps
        Kc = np.zeros((1, pairs, N_cap, w.d), np.uint16)
        Vc = np.zeros_like(Kc)
        for g in range(pairs):
            Kc[0, g, :w.N] = W.bits(W.kv_slice(w, "K", 0, g))
            Vc[0, g, :w.N] = W.bits(W.kv_slice(w, "V", 0, g))
        Pc = o.build_pyramid(Kc, N=w.N)
        seq = np.array([w.N], np.int32)
        ins = [W.decode_step_inputs(w, s, "cpu") for s in range(decode_steps)]
        t0 = time.perf_counter()
        for q, k, v in ins:
            o.decode_step(W.bits(q[:1, :pairs * w.G_Q]), W.bits(k[:1, :pairs]), W.bits(v[:1, :pairs]), Kc, Vc, Pc,
                          seq, w.K)
        per_pair = (time.perf_counter() - t0) / decode_steps / pairs
        res["decode_128k"] = {"step_us_extrapolated": per_pair * w.B * w.H_kv * 1e6,
                              "sample": f"{decode_steps} steps of {pairs} (sequence, KV head) pairs of "
                                        f"{w.B * w.H_kv}, scaled by the pair count"}
    except Exception as e:  # informational
        res["decode_128k"] = {"error": str(e)}
    return res


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import workloads as W

    w = W.WORKLOADS[args.workload]
    rows = max(16, args.cpu_sample_rows // 8)
    sample = OracleSample(w, rows * (args.steps + 1))
    for _ in range(args.warmup):
        sample.run(8)
    vals, dts = [], []
    for s in range(args.steps):
        v, dt = sample.run(rows, offset=rows * (s + 1))
        vals.append(v)
        dts.append(dt)
    value = statistics.mean(vals)
    desc = (f"per step: full pyramid + selection and attention for {rows} query positions of {w.name}, "
            f"{os.cpu_count()} threads")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": statistics.mean(dts) * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": w.name, "B": w.B, "N": w.N, "H_q": w.H_q, "H_kv": w.H_kv, "d": w.d, "K": w.K},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", "sample": desc},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_profile_section(args):
    """One measurement alone at a reduced size, for profiler captures of its kernels: the batched
    decode step with a smaller batch (the cache of 8 sequences is 2.1 GB), or the PISA and BSA
    selections at one sequence length."""
    import torch

    import workloads as W
    from hierarchical_top_block_gb300.build import build

    build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.profile_section == "decode":
        w = W.WORKLOADS["decode_128k"].with_(B=args.profile_batch)
        out = secondary_decode(w, dev, steps=args.steps, warmup=args.warmup)
    else:
        out = bsa_vs_pisa_section(dev, Ns=(args.profile_n,), steps=args.steps)
    print(json.dumps({"profile_section": args.profile_section, **out}), flush=True)


def main():
    args = parse()
    if args.profile_section:
        run_profile_section(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_pisa(args)


if __name__ == "__main__":
    main()
