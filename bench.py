#!/usr/bin/env python3
"""Benchmark of spec_verify on GB300: verified draft tokens/s and HBM GB/s.

One step = one spec_verify call over one batch of the workload (every row of
the hot path: row statistics, accept tests, residual/bonus draws, TV).  The
default workload is B = 1024 chains, k = 7, V = 151,552, bf16 logits with
independent drafts and TV output (4.66 GB of logits per step, larger than
L2, so no flush is needed between steps).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun, one rank per GPU) every rank verifies its own shard of
B chains (weak scaling, no collective on the data path); value = chains of all
ranks * k / max-over-ranks time.  Prints one JSON line on rank 0.
"""
from __future__ import annotations

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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import spec_inputs as si  # noqa: E402

METRIC = "verified draft tokens/s and HBM GB/s (% of GB300 peak) at V=151,552 bf16"
UNIT = "draft tokens/s"
CU_SOURCE = os.path.join(ROOT, "speculative_decoding_verification_68_gb300", "csrc", "spec_verify.cu")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def shard_range(rank: int, world: int, per_rank: int):
    """Chains [b0, b0 + per_rank) of the world-sized workload belong to `rank`."""
    return rank * per_rank, per_rank


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def source_sha() -> str:
    with open(CU_SOURCE, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def traffic_record(workload_name: str):
    """DRAM bytes per launch of the verification kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"sv_fused_kernel.{workload_name}.traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("source_sha256_16") != source_sha():
        return None
    return rec


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU is busy."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = [r for t, r in self.rows if t0 <= t <= t1 and len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(rows[0][2]),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


def workload_config(w: si.Workload, nb: int, world: int) -> dict:
    """The `config` object of the JSON line, identical for both arms."""
    es = 2 if w.dtype == si.BF16 else 4
    return {"workload": w.name, "batch_per_gpu": nb, "global_batch": nb * world, "k": w.k, "vocab": w.vocab,
            "logit_dtype": "bf16" if w.dtype == si.BF16 else "fp32", "tv_output": bool(w.want_tv),
            "l2": f"inputs larger than L2 ({nb * (2 * w.k + 1) * w.vocab * es / 1e9:.2f} GB of logits per step per GPU)",
            "parallelism": f"replicas x{world} (chains sharded, no collective)"}


def oracle_parity(b: si.Batch, got: dict) -> dict:
    """The GPU's outputs for batch b against the CPU oracle on the same inputs:
    chains compared, exact, decisions the oracle flagged within 1e-6 of their
    threshold (ties_flagged), chains that differ at such a tie (tie_mismatch),
    chains that differ elsewhere (beyond_band, must be 0) and the largest
    errors of p(x), q(x) and TV.  Runs outside every timed region."""
    import oracle
    from oracle import parity
    w = b.workload
    ref = oracle.default().verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, w.dtype,
                                  want_tv="tv" in got, nthreads=os.cpu_count() or 1)
    res = parity.compare({k: v.cpu().numpy() if hasattr(v, "cpu") else v for k, v in got.items()}, ref)
    res.pop("first_beyond_band", None) if res["ok"] else None
    return res


def device_batch(b: si.Batch, device):
    import torch
    if b.workload.dtype == si.BF16:
        tgt = torch.from_numpy(b.target.view(np.int16)).to(device).view(torch.bfloat16)
        dft = torch.from_numpy(b.draft.view(np.int16)).to(device).view(torch.bfloat16)
    else:
        tgt = torch.from_numpy(b.target).to(device)
        dft = torch.from_numpy(b.draft).to(device)
    return (tgt, dft, torch.from_numpy(b.tokens).to(device), torch.from_numpy(b.temperature).to(device),
            torch.from_numpy(b.uniforms).to(device))


def cpu_baseline(w: si.Workload, target_seconds: float = 10.0):
    """The CPU oracle, as it stands, on a bounded sample of chains of the workload."""
    import oracle
    orc = oracle.default()
    cores = os.cpu_count() or 1
    nb0 = min(w.batch, max(cores, 16))
    b = si.generate(w, 0, nb0)
    t = time.perf_counter()
    orc.verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, w.dtype, want_tv=w.want_tv, nthreads=cores)
    dt0 = time.perf_counter() - t
    nb = int(min(w.batch, max(nb0, nb0 * target_seconds / max(dt0, 1e-3))))
    if nb > nb0:
        b = si.generate(w, 0, nb)
    # when the whole workload takes less than the target, time it several times over
    passes = max(1, min(10, int(target_seconds / max(dt0 * nb / nb0, 1e-3))))
    t = time.perf_counter()
    for _ in range(passes):
        orc.verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, w.dtype, want_tv=w.want_tv, nthreads=cores)
    dt = (time.perf_counter() - t) / passes
    # the same oracle on one thread, over a few chains (about 1/8 of the time above)
    n1 = max(1, min(nb, int(nb * 0.125 * min(1.0, 16.0 / cores) + 0.5)))
    b1 = si.generate(w, 0, n1)
    t = time.perf_counter()
    orc.verify(b1.target, b1.draft, b1.tokens, b1.temperature, b1.uniforms, w.dtype, want_tv=w.want_tv, nthreads=1)
    dt1 = time.perf_counter() - t
    return {"value": nb * w.k / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{nb} of {w.batch} chains of {w.name} (fp64 C oracle, {cores} threads), "
                      f"{passes} pass(es) of {dt:.2f} s",
            "single_thread": {"value": n1 * w.k / dt1, "sample": f"{n1} chains on 1 thread, {dt1:.2f} s"}}


def reference_arm(args, w: si.Workload, rank: int):
    """The CPU oracle timed as the reference arm (rank 0 only)."""
    if rank != 0:
        return 0
    import oracle
    orc = oracle.default()
    cores = os.cpu_count() or 1
    nb = min(w.batch, max(cores, 16))
    b = si.generate(w, 0, nb)
    t = time.perf_counter()
    orc.verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, w.dtype, want_tv=w.want_tv, nthreads=cores)
    dt = time.perf_counter() - t
    steps_total = args.steps + args.warmup
    nb = int(min(w.batch, max(1, nb * min(4.0, 150.0 / steps_total) / max(dt, 1e-3))))
    b = si.generate(w, 0, nb)
    for _ in range(args.warmup):
        orc.verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, w.dtype, want_tv=w.want_tv, nthreads=cores)
    t = time.perf_counter()
    for _ in range(args.steps):
        orc.verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, w.dtype, want_tv=w.want_tv, nthreads=cores)
    el = time.perf_counter() - t
    value = nb * w.k * args.steps / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, w.batch, args.gpus),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{nb} of {w.batch} chains of {w.name} per step (fp64 C oracle, {cores} threads)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def measure_kernel(sv, dev_inputs, out, steps, flush=None):
    """Mean duration (ms) of the verification kernel over `steps` calls."""
    import torch
    sv.kernel_times()
    for _ in range(steps):
        if flush is not None:
            flush.zero_()
        sv.verify(*dev_inputs, out=out)
    torch.cuda.synchronize()
    kt = sv.kernel_times()
    return statistics.mean(kt), kt


REPS = 50   # timed calls per per_workload entry, L2 flushed before each


def spread_us(kt):
    """p10 / p50 / p90 of kernel durations given in ms, in microseconds."""
    q = np.percentile(np.asarray(kt, dtype=np.float64) * 1e3, [10, 50, 90])
    return {"p10": float(q[0]), "p50": float(q[1]), "p90": float(q[2]), "n": len(kt)}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=si.C5.name, choices=sorted(si.WORKLOADS))
    ap.add_argument("--batch", type=int, default=None, help="chains per GPU (default: the workload's B)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-others", action="store_true", help="skip the per-workload table")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w0 = si.WORKLOADS[args.workload]
    if args.batch is not None:
        w0 = w0.scaled(batch=args.batch, name=f"{w0.name}@B{args.batch}")

    if args.impl == "reference":
        return reference_arm(args, w0, rank)

    import torch
    import torch.distributed as dist
    import speculative_decoding_verification_68_gb300 as svlib

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    B = w0.batch
    w = w0.scaled(batch=B * world) if world > 1 else w0
    b0, nb = shard_range(rank, world, B)
    t_gen = time.perf_counter()
    batch = si.generate(w, b0, nb)
    log(f"[rank {rank}] generated {nb} chains of {w0.name} in {time.perf_counter() - t_gen:.1f} s")
    dev_in = device_batch(batch, device)
    es = 2 if w.dtype == si.BF16 else 4
    dt_name = "bf16" if w.dtype == si.BF16 else "fp32"
    sv = svlib.SpecVerifier(nb, w.k, w.vocab, dt_name, flags=svlib.SV_FLAG_KERNEL_TIMING)
    info = sv.info()
    out = sv.alloc_outputs(nb, want_pq=True, want_tv=w.want_tv, device=device)
    stream = torch.cuda.current_stream()

    # warm-up, then a short soak so the clock sampler sees the GPU under this load
    for _ in range(args.warmup):
        sv.verify(*dev_in, out=out)
    torch.cuda.synchronize()
    rc, n_bad = sv.get_error()
    if rc != 0:
        raise SystemExit(f"verification reported status {rc} ({n_bad} invalid chains) during warm-up")
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    t_soak = time.time()
    soak_end = time.time() + 1.0
    while time.time() < soak_end:
        for _ in range(50):
            sv.verify(*dev_in, out=out)
        torch.cuda.synchronize()
    sv.kernel_times()

    # ---- timed region: exactly K steps, barrier + synchronize on both sides
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        sv.verify(*dev_in, out=out)
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_wall1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    elapsed_ms = ev0.elapsed_time(ev1)
    kt = sv.kernel_times()
    if world > 1:
        tmax = torch.tensor([elapsed_ms], device=device)
        dist.all_reduce(tmax, op=dist.ReduceOp.MAX)
        elapsed_ms = float(tmax.item())
    rc, n_bad = sv.get_error()
    ms_step = elapsed_ms / args.steps
    chains_total = nb * world
    value = chains_total * w.k / (ms_step / 1e3)
    kernel_ms = statistics.mean(kt) if kt else float("nan")
    alg_bytes = nb * (2 * w.k + 1) * w.vocab * es           # per launch, per rank
    peak, peak_kind = peaks()
    achieved = alg_bytes / (kernel_ms / 1e3) / 1e9
    traffic = traffic_record(w0.name)
    tau = out["tau"].cpu().numpy()

    # ---- end to end through the public API with host buffers (pinned), copies timed
    e2e = None
    if not args.no_e2e:
        sv_h = svlib.SpecVerifier(nb, w.k, w.vocab, dt_name, flags=svlib.SV_FLAG_HOST_STAGING)
        host_in = []
        for t in dev_in:
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            host_in.append(h)
        host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out.items()}
        for _ in range(args.warmup):
            sv_h.verify_host(*host_in, out=host_out)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            sv_h.verify_host(*host_in, out=host_out)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1)
        if world > 1:
            tm = torch.tensor([e2e_ms], device=device)
            dist.all_reduce(tm, op=dist.ReduceOp.MAX)
            e2e_ms = float(tm.item())
        assert np.array_equal(host_out["tokens"].numpy(), out["tokens"].cpu().numpy())
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        e2e = {"value": chains_total * w.k / (e2e_ms / args.steps / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / args.steps,
               "api": "spec_verify_host (pinned host buffers: logits read in place over the host link)"}
        sv_h.close()
        del host_in, host_out

    # ---- the other 151,552-vocabulary workloads (kernel time, L2 flushed between calls)
    others = {}
    check = rank == 0 and world == 1 and not args.no_cpu_baseline   # the CPU leg: oracle parity counts
    if not args.no_others and rank == 0:
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
        for wo in (si.TINY, si.C2, si.C3_T0, si.C3_T06, si.C3_T1, si.C4):
            bo = si.generate(wo)
            di = device_batch(bo, device)
            so = svlib.SpecVerifier(wo.batch, wo.k, wo.vocab, "bf16" if wo.dtype == si.BF16 else "fp32",
                                    flags=svlib.SV_FLAG_KERNEL_TIMING)
            oo = so.alloc_outputs(wo.batch, want_pq=True, want_tv=True, device=device)
            for _ in range(3):
                so.verify(*di, out=oo)
            kms, kto = measure_kernel(so, di, oo, REPS, flush=flush)
            kms_warm, _ = measure_kernel(so, di, oo, REPS)   # no flush: inputs below L2 size stay resident
            ob = wo.logit_bytes
            others[wo.name] = {"kernel_us": 1e3 * kms, "kernel_us_spread": spread_us(kto),
                               "kernel_us_warm": 1e3 * kms_warm,
                               "draft_tokens_per_s": wo.batch * wo.k / (kms / 1e3),
                               "chains_per_s": wo.batch / (kms / 1e3), "gbps": ob / (kms / 1e3) / 1e9,
                               "frac_of_peak": ob / (kms / 1e3) / 1e9 / peak,
                               "accepted_tokens_per_s": float((oo["tau"].clamp(min=-1) + 1).sum().item()) / (kms / 1e3),
                               "mean_tau": float(oo["tau"].float().mean().item())}
            if check:
                others[wo.name]["parity"] = oracle_parity(bo, oo)
            so.close()
            del di, oo
        # the main workload again through spec_verify_ex: verification plus the entropy of every row
        wo = w0 if w0.batch <= 1024 else w0.scaled(batch=1024)
        bo = si.generate(wo)
        di = device_batch(bo, device)
        so = svlib.SpecVerifier(wo.batch, wo.k, wo.vocab, "bf16" if wo.dtype == si.BF16 else "fp32",
                                flags=svlib.SV_FLAG_KERNEL_TIMING)
        oo = so.alloc_outputs(wo.batch, want_pq=True, want_tv=True, device=device, want_entropy=True)
        for _ in range(3):
            so.verify(*di, out=oo)
        kms, _ = measure_kernel(so, di, oo, REPS, flush=flush)
        ob = wo.logit_bytes
        others[wo.name + "+entropy"] = {"kernel_us": 1e3 * kms, "draft_tokens_per_s": wo.batch * wo.k / (kms / 1e3),
                                        "gbps": ob / (kms / 1e3) / 1e9, "frac_of_peak": ob / (kms / 1e3) / 1e9 / peak,
                                        "api": "spec_verify_ex (entropy of every target and draft row)"}
        # ... and through spec_verify_tv: the TV of every position only (no accept tests, no bonus rows)
        otv = torch.empty((wo.batch, wo.k), dtype=torch.float32, device=device)
        for _ in range(3):
            so.verify_tv(di[0], di[1], di[3], out=otv)
        so.kernel_times()
        for _ in range(REPS):
            flush.zero_()
            so.verify_tv(di[0], di[1], di[3], out=otv)
        torch.cuda.synchronize()
        kms = statistics.mean(so.kernel_times())
        tb = wo.batch * 2 * wo.k * wo.vocab * (2 if wo.dtype == si.BF16 else 4)
        others[wo.name + "+tv_only"] = {"kernel_us": 1e3 * kms, "positions_per_s": wo.batch * wo.k / (kms / 1e3),
                                        "bytes": tb, "gbps": tb / (kms / 1e3) / 1e9,
                                        "frac_of_peak": tb / (kms / 1e3) / 1e9 / peak,
                                        "api": "spec_verify_tv (TV of every position only)"}
        so.close()
        del di, oo, bo, otv
        # a 262,144-token vocabulary (register rounds 16, one CTA per SM), independent drafts, TV on
        wo = si.Workload("b128_k7_v262144_bf16_indep_tv", 128, 7, 262144, si.BF16, 2.0, draft_mode=1,
                         draft_sigma=2.0, want_tv=True)
        bo = si.generate(wo)
        di = device_batch(bo, device)
        so = svlib.SpecVerifier(wo.batch, wo.k, wo.vocab, "bf16", flags=svlib.SV_FLAG_KERNEL_TIMING)
        oo = so.alloc_outputs(wo.batch, want_pq=True, want_tv=True, device=device)
        for _ in range(3):
            so.verify(*di, out=oo)
        kms, kto = measure_kernel(so, di, oo, REPS, flush=flush)
        ob = wo.logit_bytes
        others[wo.name] = {"kernel_us": 1e3 * kms, "kernel_us_spread": spread_us(kto),
                           "draft_tokens_per_s": wo.batch * wo.k / (kms / 1e3), "gbps": ob / (kms / 1e3) / 1e9,
                           "frac_of_peak": ob / (kms / 1e3) / 1e9 / peak, "launch": so.info()}
        so.close()
        del di, oo, bo
        # lazy verification (no TV): whole call timed with events; its bytes are the rows
        # actually read, (tau + 1) row pairs per chain, or k pairs and the bonus row
        for wo in (si.C3_T1, si.C4, w0 if w0.batch <= 1024 else w0.scaled(batch=1024)):
            bo = si.generate(wo)
            di = device_batch(bo, device)
            so = svlib.SpecVerifier(wo.batch, wo.k, wo.vocab, "bf16" if wo.dtype == si.BF16 else "fp32")
            ol = so.alloc_outputs(wo.batch, want_pq=False, device=device)
            for _ in range(3):
                so.verify_lazy(*di, out=ol)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            tot = 0.0
            for _ in range(REPS):
                flush.zero_()
                ev0.record()
                so.verify_lazy(*di, out=ol)
                ev1.record()
                torch.cuda.synchronize()
                tot += ev0.elapsed_time(ev1)
            ms = tot / REPS
            tau = np.maximum(ol["tau"].cpu().numpy().astype(np.int64), 0)
            rows = np.where(tau < wo.k, 2 * (tau + 1), 2 * wo.k + 1)
            lb = int(rows.sum()) * wo.vocab * (2 if wo.dtype == si.BF16 else 4)
            others[wo.name + "+lazy"] = {"call_us": 1e3 * ms, "draft_tokens_per_s": wo.batch * wo.k / (ms / 1e3),
                                         "chains_per_s": wo.batch / (ms / 1e3), "mean_tau": float(tau.mean()),
                                         "accepted_tokens_per_s": float((tau + 1).sum()) / (ms / 1e3),
                                         "bytes_read": lb, "gbps": lb / (ms / 1e3) / 1e9,
                                         "frac_of_peak": lb / (ms / 1e3) / 1e9 / peak,
                                         "launches_per_call": 2,
                                         "api": "spec_verify_lazy (rows past the first rejection are not read; whole call)"}
            so.close()
            del di, ol, bo
        # training side: overlap loss and its draft-logit gradient on the same workload
        wo = w0 if w0.batch <= 1024 else w0.scaled(batch=1024)
        bo = si.generate(wo)
        di = device_batch(bo, device)
        so = svlib.SpecVerifier(wo.batch, wo.k, wo.vocab, "bf16" if wo.dtype == si.BF16 else "fp32",
                                flags=svlib.SV_FLAG_KERNEL_TIMING)
        og = {"loss": torch.empty((wo.batch, wo.k), dtype=torch.float32, device=device), "grad": torch.empty_like(di[1])}
        for _ in range(3):
            so.loss_grad(di[0], di[1], di[3], kind="overlap", out=og)
        torch.cuda.synchronize()
        so.kernel_times()
        for _ in range(REPS):
            flush.zero_()
            so.loss_grad(di[0], di[1], di[3], kind="overlap", out=og)
        torch.cuda.synchronize()
        kms = statistics.mean(so.kernel_times())
        gb = 3 * wo.batch * wo.k * wo.vocab * (2 if wo.dtype == si.BF16 else 4)   # 2 rows read + 1 written per position
        others[wo.name + "+loss_grad"] = {"kernel_us": 1e3 * kms, "positions_per_s": wo.batch * wo.k / (kms / 1e3),
                                          "gbps": gb / (kms / 1e3) / 1e9, "frac_of_peak": gb / (kms / 1e3) / 1e9 / peak,
                                          "algorithmic_bytes": gb,
                                          "api": "spec_verify_loss_grad (overlap loss, gradient in the logit dtype)"}
        so.close()
        del di, og, bo
        del flush

    cpu = None
    parity_main = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        parity_main = oracle_parity(batch, out)   # the last timed step's outputs, every chain
        cpu = cpu_baseline(w0)

    if rank == 0:
        clocks = sampler.summary(t_soak, t_wall1)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == si.BF16 else "fp32", "data": "synthetic",
            "config": workload_config(w0, nb, world),
            "launch": info,
            "chains_per_s": chains_total / (ms_step / 1e3),
            "accepted_tokens_per_s": float((tau + 1).sum()) * world / (ms_step / 1e3),
            "hbm_gbps": alg_bytes * world / (ms_step / 1e3) / 1e9 / world,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": traffic["dram_bytes_per_launch"] * nb / traffic["batch"] if traffic else None,
                         "kernel": "sv_fused_kernel", "kernel_ms": kernel_ms,
                         "kernel_us_spread": spread_us(kt) if kt else None,
                         "algorithmic_bytes_per_launch": alg_bytes},
            "gpu_launches": args.steps * info["launches_per_call"],
            "clocks": clocks,
            "mean_tau": float(tau.mean()),
            "status": rc, "invalid_chains": n_bad,
            "per_workload": others,
        }
        if e2e:
            line["e2e"] = e2e
        if cpu:
            line["cpu_baseline"] = cpu
        if parity_main:
            line["parity"] = parity_main
        print(json.dumps(line), flush=True)
    sv.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
