"""Benchmark of the fused attention forward on GB300.

One step = one fused forward (O and LSE) over the long-context causal workload
B=1, H=32, Sq=Sk=65536, D=128, bf16 (inputs 1.5 GiB, larger than the 129 MB
L2, so no flush is needed between steps; workloads whose step touches less
than twice the L2 are timed step by step with the L2 flushed in between).
Throughput is TFLOP/s with the
FLOP count 4*B*H*Sq*Sk*D, halved for causal; for a sliding-window workload
(--workload window128k_causal) 4*D per visible (query, key) pair, counted
exactly.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--seed S]
                  [--heads H]   (the workload with H heads: a reduced case for profiling)
  python bench.py --impl reference ...   (the fp64 CPU oracle on a bounded sample)

Under torchrun the job is N times the workload, sharded by whole batches: rank r
processes shard r (the workload's shapes, its own seeded inputs) on its own GPU
with no cross-GPU exchange (work units are independent); the time is the max
over ranks and the value counts the work of all ranks (weak scaling).  Rank 0
prints one JSON line.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import re
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from scaled_dot_product_tcgen05_gb300 import workloads as W  # noqa: E402

DEFAULT_WORKLOAD = "long64k_causal"
PROFILE_DIR = os.path.join(ROOT, "profiles")
FALLBACK_PEAK_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 10 ** 6  # GB300 L2


# ----------------------------------------------------------------------------- ranks
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend: str):
    ws, rank, _ = dist_env()
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)
    return ws, rank


def reseed_workload(wl, seed: int):
    """The same workload with another seeded draw (seed 0: unchanged)."""
    if not 0 <= seed < 10:
        raise SystemExit("--seed must be in 0..9 (the draws of a workload family)")
    return wl if seed == 0 else dataclasses.replace(wl, draw=wl.draw + 10 * seed)


def shard_workload(wl, rank: int):
    """Shard ``rank`` of an N-times-larger job: the same shapes, its own inputs."""
    return wl if rank == 0 else dataclasses.replace(wl, draw=wl.draw + 100 * rank)


def max_over_ranks(x: float, device=None) -> float:
    """Max of a host scalar over all ranks (identity when not distributed)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def _gpu_id(self):
        try:
            u = torch.cuda.get_device_properties(self.dev).uuid
            s = str(u)
            return s if s.startswith("GPU-") else "GPU-" + s
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES")
            if vis:
                return vis.split(",")[self.dev]
            return str(self.dev)

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self._gpu_id(), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[2], parts[3:7]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, _, r in rows for i in range(4) if r[i] == "Active"})
        sm = sorted(r[0] for r in rows)
        loaded = [r for r in sm if r > 0.5 * rows[0][1]] or sm
        return {"sm_mhz": loaded[len(loaded) // 2], "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------- helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    return FALLBACK_PEAK_TFLOPS, "fallback (1.9 PFLOP/s bf16, earlier GB300 measurement)"


def fp8_peak():
    """Dense e4m3 peak: the measured bf16 peak times the nominal fp8/bf16 ratio (4.5/2.25)."""
    bf, src = peaks()
    return 2.0 * bf, src + " x 2 (nominal fp8 / bf16 dense ratio)"


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy)"
    return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


# Sources each profiled kernel is compiled from (its device code and the helpers it uses).
KERNEL_SOURCES = {
    "attn_fwd_kernel_2sm": ("ptx.cuh", "fwd_kernel.cuh", "fwd_kernel_2sm.cuh"),
    "attn_fwd_kernel": ("ptx.cuh", "fwd_kernel.cuh"),
    "attn_decode_kernel": ("ptx.cuh", "fwd_kernel.cuh", "decode_kernel.cuh"),
    "attn_bwd_kernel": ("ptx.cuh", "fwd_kernel.cuh", "bwd_kernel.cuh"),
    "attn_fwd_fp8_kernel": ("ptx.cuh", "fwd_kernel.cuh", "fwd_fp8_kernel.cuh"),
}


def source_digest(kernel: str) -> str:
    """Digest of the kernel's source files: a profile is valid only while it matches."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "scaled_dot_product_tcgen05_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def l2_flush_bytes(step_bytes: int) -> int:
    """Bytes to write between timed steps so that no input stays in L2 (0: none needed).

    A step whose buffers take at least twice the L2 evicts its own inputs before
    the next step reads them; a smaller one could find them in L2, so twice the
    L2 is written between its steps."""
    return 0 if step_bytes >= 2 * L2_BYTES else 2 * L2_BYTES


def kernel_name(D: int, decode: bool = False, causal: bool = True) -> str:
    """The kernel attn_fwd launches: CTA pairs for head dim 128 and for head dim 64
    without a causal mask, single CTAs otherwise (ATTN_PAIR=0 / 1 forces one)."""
    if decode:
        return "attn_decode_kernel"
    sel = os.environ.get("ATTN_PAIR")
    pair = sel == "1" if sel in ("0", "1") else (D == 128 or not causal)
    return "attn_fwd_kernel_2sm" if pair else "attn_fwd_kernel"


def profiled_traffic(workload: str, kernel: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it matches the sources."""
    path = os.path.join(PROFILE_DIR, f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    if not (m_t and m_h) or m_h.group(1) != source_digest(kernel):
        return None
    return float(m_t.group(1))


def workload_info(wl):
    if wl.decode:  # every cached K/V byte read once; q, o, lse
        keys = W.visible_key_counts(wl.Sk, wl.Sk, wl.causal)[wl.Sk - wl.Sq:] if wl.causal \
            else [wl.Sk] * wl.Sq
        flops = 4.0 * wl.D * wl.B * wl.H * float(sum(int(x) for x in keys))
        nbytes = (wl.B * wl.Sk * wl.H * wl.D * 2 * 2 + wl.B * wl.Sq * wl.H * wl.D * 2 * 2
                  + wl.B * wl.H * wl.Sq * 4)
        cfg = {"workload": wl.name, "B": wl.B, "H": wl.H, "Sq": wl.Sq, "Sk": wl.Sk, "D": wl.D,
               "causal": wl.causal, "dtype": wl.dtype, "decode": True, "flops_per_step": flops,
               "algorithmic_bytes_per_step": nbytes}
        return flops, nbytes, cfg
    if wl.varlen:
        lens = W.varlen_lengths(wl).tolist()
        flops = W.varlen_flops(lens, wl.H, wl.D, wl.causal)
        tokens = sum(lens)
    elif wl.backward:  # five products of 2*Sq*Sk*D per head (S^T, dP^T, dV, dK, dQ)
        flops = 2.5 * W.attention_flops(wl.B, wl.H, wl.Sq, wl.Sk, wl.D, wl.causal)
        tokens = wl.B * wl.Sq
    elif wl.windowed:  # exact count of visible (query, key) pairs
        flops = W.window_flops(wl.B, wl.H, wl.Sq, wl.Sk, wl.D, wl.causal, wl.window, wl.global_q)
        tokens = wl.B * wl.Sq
    else:
        flops = W.attention_flops(wl.B, wl.H, wl.Sq, wl.Sk, wl.D, wl.causal)
        tokens = wl.B * wl.Sq
    elem = 2
    # algorithmic bytes: read Q, K, V once, write O (16-bit) and LSE (fp32);
    # backward: read Q, K, V, O, dO and LSE, write dQ, dK, dV
    n_tensors = 8 if wl.backward else 4
    nbytes = tokens * wl.H * wl.D * elem * n_tensors + tokens * wl.H * 4
    cfg = {"workload": wl.name, "B": wl.B, "H": wl.H, "Sq": wl.Sq if not wl.varlen else tokens,
           "Sk": wl.Sk if not wl.varlen else tokens, "D": wl.D, "causal": wl.causal,
           "dtype": wl.dtype, "varlen": wl.varlen, "flops_per_step": flops,
           "algorithmic_bytes_per_step": nbytes}
    if wl.windowed:
        cfg.update(window=list(wl.window), global_q=wl.global_q)
    if wl.backward:
        cfg.update(backward=True)
    if wl.fp8:  # Q, K, V are 1 byte; O 16-bit, LSE fp32
        nbytes = tokens * wl.H * wl.D * (3 + 2) + tokens * wl.H * 4
        cfg.update(fp8="e4m3, per-tensor scales", algorithmic_bytes_per_step=nbytes)
    return flops, nbytes, cfg


def _bwd_oracle_sample(wl, n_rows=2048):
    """Head 0 of sequence 0, first n_rows positions (a causal prefix is itself a
    complete causal problem); returns (run, flops)."""
    from oracle.sdpa_oracle import attention_backward_one_head
    inp = W.make_inputs(wl, heads=[0])
    q, k, v, do = (inp[n][0, :n_rows, 0].double().numpy() for n in ("q", "k", "v", "do"))
    run = lambda: attention_backward_one_head(q, k, v, do, wl.scale, wl.causal)  # noqa: E731
    return run, 2.5 * W.attention_flops(1, 1, n_rows, n_rows, wl.D, wl.causal)


def _mask_kw(wl):
    """Oracle keyword arguments of the workload's mask."""
    return dict(window_left=wl.window[0], window_right=wl.window[1], global_q=wl.global_q)


def _row_keys(wl, rows):
    """Visible keys of the given query rows (for the sampled FLOP counts)."""
    counts = W.visible_key_counts(wl.Sq, wl.Sk, wl.causal, wl.window, wl.global_q)
    return [int(counts[i]) for i in rows]


# ------------------------------------------------------------------ reference (oracle)
def _decode_oracle_sample(wl, n_heads):
    """Inputs of the first n_heads heads of sequence 0 of a decode workload, and a
    callable running the oracle on them; returns (run, cache bytes, flops)."""
    from oracle.sdpa_oracle import attention_decode
    heads = list(range(min(n_heads, wl.H)))
    inp = W.make_inputs(wl, heads=heads)
    q, k, v = (inp[n][:1, :, heads].contiguous() for n in ("q", "k", "v"))
    run = lambda: attention_decode(q, k, v, None, wl.scale, wl.causal)  # noqa: E731
    per_head_flops, per_head_bytes, _ = workload_info(dataclasses.replace(wl, B=1, H=1))
    return run, per_head_bytes * len(heads), per_head_flops * len(heads)


def run_reference(args, wl, flops_full, cfg):
    """Times the fp64 CPU oracle, as it stands, on a bounded sample of the workload."""
    import numpy as np
    from oracle.sdpa_oracle import attention_one_head

    if wl.backward:
        run, fl = _bwd_oracle_sample(wl)
        for _ in range(args.warmup):
            run()
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            run()
            times.append(time.perf_counter() - t0)
        t = sum(times) / len(times)
        value = fl / t / 1e12
        sample = f"head 0 of {wl.name}, first 2048 positions (a complete causal sub-problem)"
        return {"metric": "attention bwd TFLOP/s", "value": value, "unit": "TFLOP/s",
                "impl": "reference", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": cfg,
                "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(),
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
    if wl.decode:
        run, nbytes, _ = _decode_oracle_sample(wl, 2)
        for _ in range(args.warmup):
            run()
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            run()
            times.append(time.perf_counter() - t0)
        t = sum(times) / len(times)
        value = nbytes / t / 1e9
        sample = f"sequence 0, heads 0-1 of {wl.name} ({nbytes:.3g} cache bytes per step)"
        return {"metric": "attention decode GB/s", "value": value, "unit": "GB/s",
                "impl": "reference", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": cfg,
                "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_threads(),
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}

    heads = list(range(min(2, wl.H)))
    S = wl.Sq
    n_rows = min(S, args.ref_rows)
    rows = sorted(set(np.linspace(0, S - 1, n_rows).astype(np.int64).tolist()))
    inp = W.make_inputs(wl, heads=heads) if not wl.varlen else W.make_inputs(wl)
    q = inp["q"][0] if not wl.varlen else inp["q"]
    k = inp["k"][0] if not wl.varlen else inp["k"]
    v = inp["v"][0] if not wl.varlen else inp["v"]
    qf = {h: q[:, h].double().numpy() for h in heads}
    kf = {h: k[:, h].double().numpy() for h in heads}
    vf = {h: v[:, h].double().numpy() for h in heads}
    sample_flops = 4.0 * wl.D * len(heads) * sum(_row_keys(wl, rows))
    times = []
    for _ in range(args.warmup):
        attention_one_head(qf[heads[0]], kf[heads[0]], vf[heads[0]], wl.scale, wl.causal,
                           rows=rows[: max(1, len(rows) // 8)], **_mask_kw(wl))
    for _ in range(args.steps):
        t0 = time.perf_counter()
        for h in heads:
            attention_one_head(qf[h], kf[h], vf[h], wl.scale, wl.causal, rows=rows,
                               **_mask_kw(wl))
        times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    value = sample_flops / t / 1e12
    cores = cpu_threads()
    sample = (f"{len(heads)} heads x {len(rows)} evenly spaced query rows of {wl.name} "
              f"(flops = 4*D*visible keys per row, {sample_flops:.3g} per step)")
    return {"metric": "attention fwd TFLOP/s", "value": value, "unit": "TFLOP/s",
            "impl": "reference", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def cpu_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_baseline_sample(wl, budget_s: float):
    """The oracle on a bounded sample of the same workload (rank 0 only)."""
    import numpy as np
    from oracle.sdpa_oracle import attention_one_head

    if wl.backward:  # a 2048-position causal prefix of head 0, repeated
        run, fl = _bwd_oracle_sample(wl)
        spent, n = 0.0, 0
        while spent < budget_s and n < 1000:
            t0 = time.perf_counter()
            run()
            spent += time.perf_counter() - t0
            n += 1
        return {"value": n * fl / spent / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(),
                "kind": "oracle",
                "sample": f"head 0, first 2048 positions of {wl.name}, {n} runs, "
                          f"{spent:.1f} s of fp64 numpy work"}
    if wl.decode:  # head 0 of sequence 0, repeated until the budget is spent
        run, nbytes, _ = _decode_oracle_sample(wl, 1)
        spent, n = 0.0, 0
        while spent < budget_s and n < 10000:
            t0 = time.perf_counter()
            run()
            spent += time.perf_counter() - t0
            n += 1
        return {"value": n * nbytes / spent / 1e9, "unit": "GB/s", "cores": cpu_threads(),
                "kind": "oracle",
                "sample": f"head 0 of sequence 0 of {wl.name}, {n} runs, "
                          f"{spent:.1f} s of fp64 numpy work"}

    inp = W.make_inputs(wl, heads=[0]) if not wl.varlen else None
    if inp is None:
        return None
    q, k, v = (inp[n][0, :, 0].double().numpy() for n in ("q", "k", "v"))
    S = wl.Sq
    done_flops, spent, n = 0.0, 0.0, 0
    chunk = 64
    rows_all = np.random.default_rng(7).permutation(S)
    t_start = time.perf_counter()
    while spent < budget_s and n < S:
        rows = sorted(rows_all[n:n + chunk].tolist())
        t0 = time.perf_counter()
        attention_one_head(q, k, v, wl.scale, wl.causal, rows=rows, **_mask_kw(wl))
        spent += time.perf_counter() - t0
        done_flops += 4.0 * wl.D * sum(_row_keys(wl, rows))
        n += chunk
    return {"value": done_flops / spent / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(),
            "kind": "oracle",
            "sample": f"{n} random query rows of head 0 of {wl.name}, "
                      f"{time.perf_counter() - t_start:.1f} s of fp64 numpy work"}


# ----------------------------------------------------------------------------- main
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--ref-rows", type=int, default=192)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--heads", type=int, default=0,
                    help="run the workload with this many heads (0: its own); reduced "
                         "cases for profiling, not the benchmark")
    ap.add_argument("--seed", type=int, default=0,
                    help="another seeded draw of the same workload (0: the standard draw)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    wl = reseed_workload(W.standard_workloads()[args.workload], args.seed)
    if args.heads:
        if not 1 <= args.heads <= wl.H:
            raise SystemExit(f"--heads must be in 1..{wl.H}")
        wl = dataclasses.replace(wl, H=args.heads)
    flops, nbytes, cfg = workload_info(wl)
    if args.seed:
        cfg = dict(cfg, seed=args.seed)
    if args.heads:
        cfg = dict(cfg, reduced_heads=args.heads)
    ws, rank, local = dist_env()

    if args.impl == "reference":
        if rank != 0:
            return 0
        cfg = dict(cfg, parallelism="replicas only (oracle on rank 0)")
        print(json.dumps(run_reference(args, wl, flops, cfg)), flush=True)
        return 0

    import scaled_dot_product_tcgen05_gb300 as pkg

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ws, rank = init_dist("nccl")
    pkg.load_library()
    wl = shard_workload(wl, rank)

    inp = W.make_inputs(wl, pin=True)
    q_h, k_h, v_h = inp["q"], inp["k"], inp["v"]
    do_h = inp.get("do")
    if wl.fp8:  # e4m3 codes (1 byte) and one scale per tensor
        (q_h, qs), (k_h, ks), (v_h, vs) = (W.quantize_e4m3(t) for t in (q_h, k_h, v_h))
        q_h, k_h, v_h = (t.view(torch.uint8).pin_memory() for t in (q_h, k_h, v_h))
    cu_h = inp["cu_seqlens_q"]
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        q, k, v = (t.to(dev, non_blocking=True) for t in (q_h, k_h, v_h))
        cu = cu_h.to(dev) if cu_h is not None else None
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev) if wl.fp8 \
            else torch.empty_like(q)
        lse_shape = (wl.H, q.shape[0]) if wl.varlen else (wl.B, wl.H, wl.Sq)
        lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
        ws_dec = None
        if wl.decode:
            need = pkg.decode_workspace_bytes(wl.B, wl.H, wl.Sq, wl.Sk, wl.D)
            ws_dec = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        if wl.fp8:
            ws_fp8 = torch.empty(pkg.fp8_workspace_bytes(wl.B, wl.H, wl.Sk, wl.D),
                                 dtype=torch.uint8, device=dev)
        if wl.backward:  # O and LSE of the forward, computed once outside the timing
            dout = do_h.to(dev, non_blocking=True)
            pkg.attn_fwd(q, k, v, causal=wl.causal, scale=wl.scale, out=o, lse=lse,
                         stream=stream)
            ws_bwd = torch.empty(pkg.bwd_workspace_bytes(wl.B, wl.H, wl.Sq, wl.D),
                                 dtype=torch.uint8, device=dev)
            dq_t, dk_t, dv_t = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    torch.cuda.synchronize()

    # one set of device buffers; the end-to-end leg uses a second one as well
    bs0 = dict(q=q, k=k, v=v, o=o, lse=lse)
    if wl.backward:
        bs0.update(dout=dout, dq=dq_t, dk=dk_t, dv=dv_t)

    def run_step(bs):
        if wl.fp8:
            pkg.attn_fwd_fp8(bs["q"], bs["k"], bs["v"], q_scale=qs, k_scale=ks, v_scale=vs,
                             causal=wl.causal, scale=wl.scale, workspace=ws_fp8, out=bs["o"],
                             lse=bs["lse"], stream=stream)
            return
        if wl.backward:
            pkg.attn_bwd(bs["q"], bs["k"], bs["v"], bs["o"], bs["dout"], bs["lse"],
                         causal=wl.causal, scale=wl.scale, workspace=ws_bwd, dq=bs["dq"],
                         dk=bs["dk"], dv=bs["dv"], stream=stream)
            return
        if wl.decode:
            pkg.attn_decode(bs["q"], bs["k"], bs["v"], causal=wl.causal, scale=wl.scale,
                            workspace=ws_dec, out=bs["o"], lse=bs["lse"], stream=stream)
            return
        pkg.attn_fwd(bs["q"], bs["k"], bs["v"], causal=wl.causal, scale=wl.scale,
                     cu_seqlens_q=cu, cu_seqlens_k=cu, out=bs["o"], lse=bs["lse"],
                     window=wl.window, global_q=wl.global_q, stream=stream)

    def step():
        run_step(bs0)

    # ---- kernel-only timed region (inputs resident in HBM)
    for _ in range(args.warmup):
        step()
    st = pkg.attn_check(stream)
    if st != pkg.ATTN_OK:
        raise SystemExit(f"device status {pkg.status_string(st)}")
    grid, smem = pkg.last_launch()
    launches_per_step = 3 if wl.backward else 1  # backward: D pre-pass, main, dQ conversion
    if wl.fp8:
        launches_per_step = 2  # V transpose, attention
    if wl.decode and pkg.decode_workspace_bytes(wl.B, wl.H, wl.Sq, wl.Sk, wl.D) > 0:
        launches_per_step = 2  # the split decode kernel and the merge kernel
    # Inputs that could stay in L2 from one step to the next are evicted between
    # timed steps by writing a buffer twice the L2's size; each step is then timed
    # alone (its own pair of events) and the flush stays outside the timed steps.
    step_bytes = sum(t.numel() * t.element_size() for t in bs0.values())
    flush_bytes = l2_flush_bytes(step_bytes)
    flush = None
    if flush_bytes:
        flush = torch.empty(flush_bytes, dtype=torch.uint8, device=dev)
    sampler = ClockSampler(local)
    sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    st = pkg.attn_check(stream)
    if st != pkg.ATTN_OK:
        raise SystemExit(f"device status {pkg.status_string(st)}")
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    if flush is None:  # back to back: the whole region
        total_ms = ev[0][0].elapsed_time(ev[-1][1])
    else:  # the steps alone, without the flushes between them
        total_ms = sum(launch_ms)
    ms_step = max_over_ranks(total_ms / args.steps, dev)
    kernel_ms = sum(launch_ms) / len(launch_ms)
    l2_note = ("no flush: a step touches %.2f GiB > twice the %d MB L2" %
               (step_bytes / 2 ** 30, L2_BYTES // 10 ** 6) if flush is None else
               "L2 flushed between timed steps (%d MB written; a step touches %.1f MB)" %
               (flush_bytes // 10 ** 6, step_bytes / 1e6))
    del flush

    # ---- end to end through the public API, host buffers, copies inside the region
    o_h = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    lse_h = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    if wl.backward:  # inputs q, k, v, o, dO, LSE in; dQ, dK, dV out
        with torch.cuda.stream(stream):
            o_h.copy_(o, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)
        torch.cuda.synchronize()
        g_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq_t, dk_t, dv_t)]

    # Double-buffered: step i uploads its inputs into buffer set i % 2 on one
    # copy stream while step i - 1 computes, and downloads its results on
    # another; a set is refilled only after its previous results have left.
    with torch.cuda.stream(stream):
        bs1 = {name: torch.empty_like(t) for name, t in bs0.items()}
    torch.cuda.synchronize()
    sets = (bs0, bs1)
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    host_in = [("q", q_h), ("k", k_h), ("v", v_h)]
    if wl.backward:  # inputs q, k, v, o, dO, LSE in; dQ, dK, dV out
        host_in += [("o", o_h), ("lse", lse_h), ("dout", do_h)]
        host_out = list(zip(g_h, ("dq", "dk", "dv")))
    else:
        host_out = [(o_h, "o"), (lse_h, "lse")]
    freed = [None, None]

    def e2e_steps(n):
        for i in range(n):
            bs = sets[i % 2]
            if freed[i % 2] is not None:
                up.wait_event(freed[i % 2])
            with torch.cuda.stream(up):
                for name, h in host_in:
                    bs[name].copy_(h, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(up)
            stream.wait_event(ready)
            run_step(bs)
            done = torch.cuda.Event()
            done.record(stream)
            down.wait_event(done)
            with torch.cuda.stream(down):
                for h, name in host_out:
                    h.copy_(bs[name], non_blocking=True)
            freed[i % 2] = torch.cuda.Event()
            freed[i % 2].record(down)

    e2e_steps(args.warmup)
    torch.cuda.synchronize()
    e_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    barrier()
    torch.cuda.synchronize()
    freed = [None, None]
    e_ev[0].record(up)
    e2e_steps(args.steps)
    down.wait_event(freed[(args.steps - 1) % 2])
    e_ev[1].record(down)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(e_ev[0].elapsed_time(e_ev[1]) / args.steps, dev)
    if not (torch.isfinite(o_h.float()).all() and torch.isfinite(lse_h).all()):
        raise SystemExit("non-finite output")
    h2d = (q_h.numel() + k_h.numel() + v_h.numel()) * q_h.element_size()
    d2h = o_h.numel() * o_h.element_size() + lse_h.numel() * 4
    if wl.backward:
        h2d += (o_h.numel() + do_h.numel()) * q_h.element_size() + lse_h.numel() * 4
        d2h = sum(t.numel() for t in g_h) * q_h.element_size()
        if not all(torch.isfinite(t.float()).all() for t in g_h):
            raise SystemExit("non-finite gradient")

    if rank != 0:
        return 0
    if wl.decode:  # HBM-bound: bytes per step against the measured copy bandwidth
        peak, peak_src = hbm_peak()
        achieved = nbytes / (kernel_ms * 1e-3) / 1e9
        kern = kernel_name(wl.D, decode=True)
        per_step = nbytes * ws / 1e9
        unit, metric, bound = "GB/s", "attention decode GB/s", "hbm"
    else:
        peak, peak_src = peaks()
        achieved = flops / (kernel_ms * 1e-3) / 1e12
        kern = kernel_name(wl.D, causal=wl.causal)
        per_step = flops * ws / 1e12
        unit, metric, bound = "TFLOP/s", "attention fwd TFLOP/s", "tensor"
        if wl.backward:
            kern = "attn_bwd_kernel"
            metric = "attention bwd TFLOP/s"
        if wl.fp8:
            peak, peak_src = fp8_peak()
            achieved = flops / (kernel_ms * 1e-3) / 1e12
            kern = "attn_fwd_fp8_kernel"
            metric = "attention fwd fp8 TFLOP/s"
    traffic = None if args.heads else profiled_traffic(wl.name, kern)  # a full launch's bytes
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample(wl, args.cpu_budget_s)
    cfg = dict(cfg, parallelism=f"dp{ws}: rank r processes shard r (own inputs)" if ws > 1
               else "single GPU",
               l2=l2_note,
               grid_ctas=grid, smem_bytes=smem)
    out = {
        "metric": metric, "value": per_step / (ms_step * 1e-3),
        "unit": unit, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if wl.fp8 else ("bf16" if wl.dtype == "bf16" else "fp16"),
        "data": "synthetic", "config": cfg,
        "pct_of_peak": achieved / peak,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src,
                     "kernel": kern, "kernel_ms": kernel_ms},
        "e2e": {"value": per_step / (e2e_ms * 1e-3), "unit": unit,
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "overlap": "double-buffered: step i+1's upload and step i-1's download run "
                           "on two copy streams while step i computes"},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
