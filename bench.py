"""Benchmark: decode effective weight GB/s & tok/s of the fused dual-path
kernel on one Llama-style decoder block at 8B shape (q8_0 base + rank-16 LoRA,
s = 2.0, on all seven projections, batch-1 decode, bf16 activations).

One step = one decode token through the block, launched as a decoder block
launches it: q, k and v in one multi-tensor call (they share the input), o,
gate and up in one multi-tensor call, down.  Each projection consumes a seeded
bf16 activation of its own d_in.  value = effective weight bytes (quantized base incl. scales + LoRA A/B)
per step / device time per step; tok/s = steps / s.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no data exchange); the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth as S  # noqa: E402

METRIC = "decode effective weight GB/s & tok/s (8B shape, q8_0+LoRA) vs HBM peak"
WORKLOAD = ("8B-shape decoder block: q,o 4096x4096; k,v 1024x4096; gate,up 14336x4096; down 4096x14336; "
            "q8_0 base ~N(0,0.02); rank-16 LoRA ~N(0,0.01), s=2.0 on all 7; batch-1 decode; x bf16 ~N(0,1)")
RANK = 16
SCALE = 2.0
N_COPIES = 3


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def effective_bytes(base, ad):
    """Per step: qs + d planes of all tensors, plus A and B of the adapter."""
    tot = 0
    for t in base.tensors:
        tot += S.qs_bytes(base.quant, t.d_out, t.d_in) + S.d_bytes(t.d_out, t.d_in)
        tot += RANK * t.d_in * 4 + t.d_out * RANK * 4
    return tot


def algorithmic_bytes(base, ad):
    """Effective bytes plus x (bf16) read and y (fp32) written."""
    return effective_bytes(base, ad) + sum(t.d_in * 2 + t.d_out * 4 for t in base.tensors)


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
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
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- oracle legs
def oracle_dual_step(base, ad, xs, proj):
    import oracle as O
    qs, d = base.planes[proj]
    deq = O.dequantize(base.quant, qs, d)
    A, B = ad.factors[proj]
    return O.dual_path(deq, [(A, B, SCALE)], xs[base.tensors[proj].d_in])


def proj_effective_bytes(base, proj):
    t = base.tensors[proj]
    return S.qs_bytes(base.quant, t.d_out, t.d_in) + S.d_bytes(t.d_out, t.d_in) + RANK * (t.d_in + t.d_out) * 4


def cpu_baseline(base, ad, xs, budget_s=12.0):
    """The oracle as it stands on the host cores: whole projections of the
    block in order until ~budget_s of work; GB/s on the same byte count."""
    done_bytes, t0, n = 0, time.perf_counter(), 0
    while True:
        p = n % 7
        oracle_dual_step(base, ad, xs, p)
        done_bytes += proj_effective_bytes(base, p)
        n += 1
        el = time.perf_counter() - t0
        if el > budget_s:
            break
    return {"value": done_bytes / el / 1e9, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} projection calls (q, k, v, o, gate, up, down in turn) of the same block, fp64 numpy oracle "
                      f"(dequantize + GEMV + low-rank), {el:.1f} s; numpy BLAS may use all {os.cpu_count()} cores"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    base = S.block_base(S.Q8_0)
    ad = S.block_adapter(base, adapter=0, rank=RANK)
    xs = {d: S.bf16_bits_to_f32(S.to_bf16_bits(S.activations(1, d))).astype(np.float64) for d in (4096, 14336)}
    for i in range(args.warmup):
        oracle_dual_step(base, ad, xs, i % 7)
    tot_bytes, t0 = 0, time.perf_counter()
    for i in range(args.steps):
        oracle_dual_step(base, ad, xs, i % 7)
        tot_bytes += proj_effective_bytes(base, i % 7)
    el = time.perf_counter() - t0
    val = tot_bytes / el / 1e9
    sample = (f"{args.steps} steps, step i = one projection ({'/'.join(S.PROJ)} in turn) of the block through "
              f"the fp64 numpy oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": "one projection per step"},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ---------------------------------------------------------------- GPU leg
def run_ours(args, world, rank, local):
    import torch
    import quantized_base_lora_gb300 as q
    from quantized_base_lora_gb300.runtime import Runtime

    torch.cuda.set_device(local)
    base = S.block_base(S.Q8_0)
    ad = S.block_adapter(base, adapter=0, rank=RANK)
    tt = [(t.layer, t.proj, t.d_out, t.d_in, t.qs_off, t.d_off) for t in base.tensors]
    digest, ad_digest = S.content_digest(base.buf), S.content_digest(ad.payload)
    # N_COPIES contexts over identical base copies: consecutive steps read
    # different HBM (3 x 231.7 MB > 129 MB L2), so no step is L2-resident.
    rts = []
    for c in range(N_COPIES):
        rt = Runtime(arena_bytes=64 << 20)
        q.check(rt.load_base(base.quant, tt, base.buf, digest), rt.ctx)
        st, h = rt.stage(ad, ad_digest)
        q.check(st, rt.ctx)
        q.check(rt.activate([h], [SCALE])[0], rt.ctx)
        rts.append(rt)
    dev = torch.device("cuda", local)
    xs_host = {d: S.to_bf16_bits(S.activations(1, d)) for d in (4096, 14336)}
    xs = {d: torch.from_numpy(v.view(np.int16)).to(dev).view(torch.bfloat16) for d, v in xs_host.items()}
    d_outs = [t.d_out for t in base.tensors]
    y_off = np.concatenate([[0], np.cumsum(d_outs)]).astype(int)
    ybuf = torch.empty(int(y_off[-1]), dtype=torch.float32, device=dev)
    x_addr = {d: v.data_ptr() for d, v in xs.items()}
    stream = torch.cuda.Stream(device=dev)
    sh = int(stream.cuda_stream)

    groups = [[0, 1, 2], [3], [4, 5], [6]]          # qkv | o | gate+up | down

    y_ptr = [ybuf.data_ptr() + 4 * int(y_off[i]) for i in range(len(d_outs))]

    def step(rt, xmap):
        # xmap: d_in -> device address of that step's activations (bf16)
        for grp in groups:
            xp = xmap[base.tensors[grp[0]].d_in]
            if len(grp) == 1:
                st = q.ovl_linear_forward(rt.ctx, grp[0], xp, q.OVL_BF16, 1, y_ptr[grp[0]], q.OVL_PATH_DUAL, 0, 0, sh)
            else:
                st = q.ovl_linear_forward_multi(rt.ctx, grp, xp, q.OVL_BF16, 1, [y_ptr[i] for i in grp], sh)
            if st != 0:
                raise q.OvlError(st, q.ovl_last_error(rt.ctx))

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(rts[i % N_COPIES], x_addr)
    stream.synchronize()
    for rt in rts:
        q.check(q.ovl_check_device(rt.ctx, sh), rt.ctx)

    # ---- device-resident timed region
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    # One event pair around the whole region: an event recorded between two
    # launches would cut the programmatic dependency that lets each launch's
    # CTAs start streaming while the previous grid drains.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(args.steps):
            step(rts[i % N_COPIES], x_addr)
        ev1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    clocks = clk.stop()
    total_ms = ev0.elapsed_time(ev1)
    for rt in rts:
        q.check(q.ovl_check_device(rt.ctx, sh), rt.ctx)

    # ---- end to end: pinned host x in, host y out, every step
    x_pin = {d: torch.from_numpy(v.view(np.int16)).pin_memory() for d, v in xs_host.items()}
    x_dev = {d: torch.empty(v.shape, dtype=torch.int16, device=dev) for d, v in xs_host.items()}
    xdev_addr = {d: v.data_ptr() for d, v in x_dev.items()}
    y_pin = torch.empty(int(y_off[-1]), dtype=torch.float32).pin_memory()
    h2d = sum(v.nbytes for v in xs_host.values())
    d2h = int(y_off[-1]) * 4
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.steps):
            for d in x_dev:
                x_dev[d].copy_(x_pin[d], non_blocking=True)
            step(rts[i % N_COPIES], xdev_addr)
            y_pin.copy_(ybuf, non_blocking=True)
        e1.record(stream)
    stream.synchronize()
    e2e_ms = e0.elapsed_time(e1)

    eff = effective_bytes(base, ad)
    alg = algorithmic_bytes(base, ad)
    t_max = max_over_ranks(total_ms, world)
    e2e_max = max_over_ranks(e2e_ms, world)
    if rank != 0:
        return
    peak, peak_kind = peaks()
    mean_step_s = total_ms / args.steps / 1e3
    achieved = alg / mean_step_s / 1e9
    value = world * eff * args.steps / (t_max / 1e3) / 1e9
    out = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": t_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "s8xs8->s32 dp4a + f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": world, "seq_len": 1, "parallelism": f"replicas x{world}",
                   "l2": f"{N_COPIES} identical base copies rotated per step ({N_COPIES} x "
                         f"{eff / 1e6:.1f} MB > 129 MB L2); no flush inside the timed region",
                   "effective_bytes_per_step": eff, "algorithmic_bytes_per_step": alg},
        "tok_s": world * args.steps / (t_max / 1e3),
        "tok_s_per_gpu": args.steps / (t_max / 1e3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "k_dualpath (4 launches per step: qkv, o, gate+up, down)",
                     "note": f"peak = {peak_kind} HBM copy bandwidth; achieved = algorithmic bytes per step / mean "
                             f"step, CUDA events on the launching stream around the timed region (a step is "
                             f"only k_dualpath launches)"},
        "e2e": {"value": world * eff * args.steps / (e2e_max / 1e3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": len(groups) * args.steps,
        "clocks": clocks,
    }
    if world == 1:
        xs64 = {d: S.bf16_bits_to_f32(v).astype(np.float64) for d, v in xs_host.items()}
        out["cpu_baseline"] = cpu_baseline(base, ad, xs64)
    print(json.dumps(out))
    for rt in rts:
        rt.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    args = ap.parse_args()
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
