"""Benchmark: decode effective weight GB/s & tok/s of the fused dual-path
kernel on one Llama-style decoder block at 8B shape (q8_0 base + rank-16 LoRA,
s = 2.0, on all seven projections, batch-1 decode, bf16 activations).

One step = one decode token through the block, launched as a decoder block
launches it: q, k and v in one multi-tensor call (they share the input), o,
gate and up in one multi-tensor call, down.  Each projection consumes a seeded
bf16 activation of its own d_in.  value = effective weight bytes (quantized base incl. scales + LoRA A/B)
per step / device time per step; tok/s = steps / s.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                      [--workload decode|q4-stacked|segmented|jit-prefill|decode32|switch]
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no data exchange); the slowest rank's time is used.

--workload selects the other measured configurations (one GPU, one JSON line
each; the default, decode, is the headline line above):
  q4-stacked   8B-shape q4_0 block, stacked rank-16 (s=1) + rank-64 (s=0.5)
               adapters, dual path at T = 1, 4, 8
  segmented    64 decode requests over 16 rank-16 adapters (TABLE, Zipf 1.1),
               q4_0 q (4096x4096) and gate (14336x4096)
  jit-prefill  one 8B-shape q8_0 layer + rank-16 adapter, T = 512 prefill on the
               per-layer JIT path (fp32 materialization + tcgen05 TF32 GEMM)
  decode32     32 layers of the 8B block (q8_0 + rank-16 on all 224 tensors),
               batch-1 decode, tokens/s
  switch       activate / rollback latency over four 32-layer adapters
               (168 MB each, one with a corrupt declared digest)
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


# DRAM bytes (read + write) per k_dualpath launch of the decode step, mean over
# its four launches, measured by ncu with --metrics dram__bytes_read.sum,
# dram__bytes_write.sum on this workload.  None whenever k_dualpath has changed
# since the counters were taken, until it is measured again.
K1_TRAFFIC_PER_LAUNCH = 59_391_104


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
                      f"(dequantize + GEMV + low-rank), {el:.1f} s; numpy BLAS may use all {os.cpu_count()} cores, "
                      f"the elementwise dequantization runs on one"}


def cpu_baseline_one_thread(budget_s=10.0):
    """The same oracle leg in a child process whose BLAS runs one thread (the
    thread count of numpy's BLAS is fixed when it loads, so it is set in the
    child's environment)."""
    code = ("import json, sys; sys.path.insert(0, %r); import numpy as np; import synth as S; import bench; "
            "base = S.block_base(S.Q8_0); ad = S.block_adapter(base, adapter=0, rank=bench.RANK); "
            "xs = {d: S.bf16_bits_to_f32(S.to_bf16_bits(S.activations(1, d))).astype(np.float64) "
            "for d in (4096, 14336)}; print(json.dumps(bench.cpu_baseline(base, ad, xs, budget_s=%r)))"
            % (ROOT, budget_s))
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1")
    try:
        p = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        out = json.loads(p.stdout.strip().splitlines()[-1])
        out["cores"] = 1
        out["sample"] = out["sample"].split("; numpy BLAS")[0] + "; every BLAS pool limited to one thread"
        return out
    except Exception as e:   # reported, not fatal: the all-core figure stands
        return {"value": None, "cores": 1, "kind": "oracle", "error": str(e)[:200]}


def run_reference(args, world, rank):
    if rank != 0:
        return
    # Step i runs projection i mod 7; a run of fewer than 7 steps builds only the
    # projections it uses (every projection has its own seeds, so they are the
    # same bytes as in the whole block).
    n_proj = min(7, max(1, args.steps, args.warmup))
    base = S.block_base(S.Q8_0, projs=S.PROJ[:n_proj])
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
    stream = torch.cuda.Stream(device=dev)
    sh = int(stream.cuda_stream)
    step = block_step(q, base.tensors, sh)
    x_addr = {d: v.data_ptr() for d, v in xs.items()}
    y_ptr = [ybuf.data_ptr() + 4 * int(y_off[i]) for i in range(len(d_outs))]

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(rts[i % N_COPIES], x_addr, y_ptr)
    stream.synchronize()
    for rt in rts:
        q.check(q.ovl_check_device(rt.ctx, sh), rt.ctx)

    # ---- device-resident timed regions: REPEATS regions of exactly K steps,
    # each bracketed by a barrier and a synchronize and timed by one event pair
    # on the launching stream (an event between two launches would cut the
    # programmatic dependency that lets a launch stream while the previous
    # grid drains); the median region is the reported one.
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)

    def one_region(i0):
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                step(rts[(i0 + i) % N_COPIES], x_addr, y_ptr)

    region_ms = timed_regions(one_region, stream, world)
    clocks = clk.stop()
    for rt in rts:
        q.check(q.ovl_check_device(rt.ctx, sh), rt.ctx)

    # ---- end to end through the same C-ABI calls: every step stages its x
    # from page-locked host memory and its y lands in page-locked host memory
    e2e_ms, h2d, d2h = e2e_region(torch, q, step, rts, xs_host, int(y_off[-1]), y_off, stream, dev, args.steps)

    # ---- tok/s: one decode token through the 32-layer stack of the block,
    # every layer with its own seeds (224 projection calls, 128 launches)
    tok = decode32_tok_s(args, q, torch, dev, stream) if world == 1 else None

    eff = effective_bytes(base, ad)
    alg = algorithmic_bytes(base, ad)
    med_ms = statistics.median(region_ms)
    t_max = max_over_ranks(med_ms, world)
    e2e_max = max_over_ranks(e2e_ms, world)
    if rank != 0:
        return
    peak, peak_kind = peaks()
    mean_step_s = med_ms / args.steps / 1e3
    achieved = alg / mean_step_s / 1e9
    value = world * eff * args.steps / (t_max / 1e3) / 1e9
    mhz = clocks.get("sm_mhz") or 0.0
    out = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": t_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "s8xs8->s32 dp4a + f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": world, "seq_len": 1, "parallelism": f"replicas x{world}",
                   "l2": f"{N_COPIES} identical base copies rotated per step ({N_COPIES} x "
                         f"{eff / 1e6:.1f} MB > 129 MB L2); no flush inside the timed region",
                   "effective_bytes_per_step": eff, "algorithmic_bytes_per_step": alg,
                   "timing": f"{REPEATS} regions of {args.steps} steps each; value from the median region"},
        "repeats": {"ms_per_step": [r / args.steps for r in region_ms],
                    "us_per_step_x_sm_mhz": [r / args.steps * 1e3 * mhz for r in region_ms],
                    "sm_mhz_median": mhz},
        "tok_s": tok["tok_s"] if tok else None,
        "tok_s_note": ("decode tokens/s through the 32-layer stack of the block (every layer its own seeds, "
                       "rank-16 LoRA on all 224 projections), 1 / time of one token's 224 projection calls; "
                       "measured at N=1 only") if tok else "measured at N=1 only",
        "tok_s_detail": tok,
        "block_steps_per_s": world * args.steps / (t_max / 1e3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": K1_TRAFFIC_PER_LAUNCH,
                     "algorithmic_bytes_per_launch": alg / len(GROUPS),
                     "traffic_note": "dram__bytes_read.sum + dram__bytes_write.sum per k_dualpath launch, mean over "
                                     "the step's launches, from one ncu capture of this kernel build on this workload",
                     "kernel": "k_dualpath (4 launches per step: qkv, o, gate+up, down)",
                     "note": f"peak = {peak_kind} HBM copy bandwidth; achieved = algorithmic bytes per step / step "
                             f"time of the median region, CUDA events on the launching stream (a step is only "
                             f"k_dualpath launches)"},
        "e2e": {"value": world * eff * args.steps / (e2e_max / 1e3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "per step: ovl_stage_activations of both activations (page-locked host -> device, one "
                       "kernel in the programmatic launch chain), then the 4 forward calls with y in page-locked "
                       f"host memory; median of {REPEATS} regions of {args.steps} steps"},
        "gpu_launches": len(GROUPS) * args.steps * REPEATS,
        "clocks": clocks,
    }
    for rt in rts:
        rt.close()
    if world == 1:
        xs64 = {d: S.bf16_bits_to_f32(v).astype(np.float64) for d, v in xs_host.items()}
        out["cpu_baseline"] = cpu_baseline(base, ad, xs64)
        out["cpu_baseline"]["one_thread"] = cpu_baseline_one_thread()
        out["secondary"] = secondary_workloads(args)
    print(json.dumps(out))


SECONDARY = ("q4k-decode", "q4-stacked", "prefill-dual", "segmented")


def secondary_workloads(args):
    """The other workloads' key figures in the same run (50 steps each after 5
    warm-up steps, median of REPEATS regions; each its own timed regions, none
    inside the headline's): the line each `--workload` prints, reduced to its
    value, step time and roofline fraction per token count."""
    res = {}
    sargs = argparse.Namespace(**{**vars(args), "steps": 50, "warmup": 5})
    global emit
    keep = emit
    for name in SECONDARY:
        got = []
        emit = got.append
        try:
            WORKLOADS[name](sargs)
        except Exception as e:   # reported, not fatal: the headline stands
            got = [{"error": f"{type(e).__name__}: {e}"[:200]}]
        finally:
            emit = keep
        line = got[-1] if got else {}
        entry = {k: line.get(k) for k in ("metric", "value", "unit", "error") if line.get(k) is not None}
        if "per_T" in line:
            entry["per_T"] = {str(T): {"us_per_step": round(v["ms_per_step"] * 1e3, 2),
                                       "frac": round(v["roofline"]["frac"], 4),
                                       "bound": v["roofline"]["bound"]} for T, v in line["per_T"].items()}
        elif "roofline" in line:
            entry["frac"] = round(line["roofline"]["frac"], 4)
            entry["bound"] = line["roofline"]["bound"]
        res[name] = entry
    return res


GROUPS = [[0, 1, 2], [3], [4, 5], [6]]          # qkv | o | gate+up | down
REPEATS = 5


def block_step(q, tensors, sh, layer_base: int = 0):
    """One decode step of a block: q+k+v, o, gate+up, down (four calls, the
    multi-tensor ones for tensors that share x).  step(rt, x_addr, y_ptr):
    x_addr maps d_in to the device address of that step's bf16 activations,
    y_ptr[i] is the output of tensor i of the block."""
    def step(rt, x_addr, y_ptr, layer_base=layer_base):
        for grp in GROUPS:
            xp = x_addr[tensors[grp[0]].d_in]
            if len(grp) == 1:
                st = q.ovl_linear_forward(rt.ctx, layer_base + grp[0], xp, q.OVL_BF16, 1, y_ptr[grp[0]],
                                          q.OVL_PATH_DUAL, 0, 0, sh)
            else:
                st = q.ovl_linear_forward_multi(rt.ctx, [layer_base + i for i in grp], xp, q.OVL_BF16, 1,
                                                [y_ptr[i] for i in grp], sh)
            if st != 0:
                raise q.OvlError(st, q.ovl_last_error(rt.ctx))
    return step


def timed_regions(one_region, stream, world, repeats=REPEATS):
    """Device ms of `repeats` regions, each one call of one_region(start index)
    between a barrier + synchronize on both sides, timed by one event pair on
    `stream`."""
    import torch
    out = []
    for r in range(repeats):
        barrier(world)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        one_region(r)
        ev1.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        barrier(world)
        out.append(ev0.elapsed_time(ev1))
    return out


def e2e_region(torch, q, step, rts, xs_host, n_y, y_off, stream, dev, steps):
    """End-to-end ms of `steps` steps through the public C ABI: every step
    stages its activations (both d_in, one page-locked host buffer) into the
    device with ovl_stage_activations, whose kernel joins the programmatic
    launch chain, and the step's calls write y straight into page-locked host
    memory (two host buffers, alternating)."""
    x_cat = np.concatenate([xs_host[d].reshape(-1) for d in (4096, 14336)])
    x_pin = torch.from_numpy(x_cat.view(np.int16)).pin_memory()
    x_dev = torch.empty(x_pin.shape, dtype=torch.int16, device=dev)
    y_pin = [torch.empty(n_y, dtype=torch.float32).pin_memory() for _ in range(2)]
    x_addr = {4096: x_dev.data_ptr(), 14336: x_dev.data_ptr() + 4096 * 2}
    y_ptr = [[yb.data_ptr() + 4 * int(y_off[i]) for i in range(len(y_off) - 1)] for yb in y_pin]
    h2d = x_cat.nbytes
    d2h = n_y * 4
    sh = int(stream.cuda_stream)

    def one(i):
        st = q.ovl_stage_activations(x_dev.data_ptr(), x_pin.data_ptr(), h2d, sh)
        if st != 0:
            raise q.OvlError(st, "stage activations")
        step(rts[i % len(rts)], x_addr, y_ptr[i % 2])

    with torch.cuda.stream(stream):
        for i in range(3):
            one(i)
    stream.synchronize()

    def region(r):
        with torch.cuda.stream(stream):
            for i in range(steps):
                one(r * steps + i)

    ms = timed_regions(region, stream, 1)
    return statistics.median(ms), h2d, d2h


def decode32_tok_s(args, q, torch, dev, stream):
    """Tokens/s of one decode token through LAYERS layers of the 8B-shape block
    (q8_0, every layer with its own seeds, ~7.4 GB), a rank-16 adapter (own
    seeds per layer and projection, s = 2.0) on all 224 projections."""
    from quantized_base_lora_gb300.runtime import Runtime
    from synth.stack import layer_stride, stack_adapter
    rt = Runtime(arena_bytes=256 << 20)
    stride = layer_stride(S.Q8_0)
    stack = load_stack(rt, torch, dev)
    ad = stack_adapter(stack, adapter=0, rank=RANK)
    st, h = rt.stage(ad, S.content_digest(ad.payload))
    q.check(st, rt.ctx)
    q.check(rt.activate([h], [SCALE])[0], rt.ctx)
    sh = int(stream.cuda_stream)
    one = stack.tensors[:7]
    xs = {d: torch.from_numpy(S.to_bf16_bits(S.activations(1, d)).view(np.int16)).to(dev).view(torch.bfloat16)
          for d in (4096, 14336)}
    x_addr = {d: v.data_ptr() for d, v in xs.items()}
    ys = [torch.empty((1, t.d_out), dtype=torch.float32, device=dev) for t in one]
    y_ptr = [y.data_ptr() for y in ys]
    step = block_step(q, one, sh)
    n = len(one)

    def token():
        for l in range(LAYERS):
            step(rt, x_addr, y_ptr, layer_base=l * n)

    with torch.cuda.stream(stream):
        for _ in range(3):
            token()
    stream.synchronize()
    q.check(q.ovl_check_device(rt.ctx, sh), rt.ctx)
    k = max(3, min(args.steps, 20))

    def region(_):
        with torch.cuda.stream(stream):
            for _ in range(k):
                token()

    ms = timed_regions(region, stream, 1)
    q.check(q.ovl_check_device(rt.ctx, sh), rt.ctx)
    one_block = S.Base(S.Q8_0, one, np.zeros(0, np.uint8))
    alg = LAYERS * algorithmic_bytes(one_block, None)
    med = statistics.median(ms) / k
    peak, kind = peaks()
    rt.close()
    rt.base = None
    torch.cuda.empty_cache()
    return {"tok_s": 1e3 / med, "ms_per_token": med, "tokens_per_region": k,
            "repeats_ms_per_token": [m / k for m in ms],
            "launches_per_token": LAYERS * len(GROUPS),
            "roofline": {"bound": "hbm", "achieved": alg / (med / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": alg / (med / 1e3) / 1e9 / peak, "algorithmic_bytes_per_token": alg,
                         "note": f"peak = {kind} HBM copy bandwidth"},
            "base": f"{LAYERS} layers x 231.7 MB q8_0 ({LAYERS * stride / 1e9:.2f} GB incl. 64 KiB padding)"}


# ---------------------------------------------------------------- other workloads
def timed_steps(step, steps, warmup, stream):
    """Median device ms per step over REPEATS regions of `steps` steps (after
    the warm-up), each region timed by one event pair on `stream`."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            step(i)
    stream.synchronize()

    def region(r):
        with torch.cuda.stream(stream):
            for i in range(steps):
                step(r * steps + i)

    return statistics.median(timed_regions(region, stream, 1)) / steps


def emit(line: dict):
    print(json.dumps(line), flush=True)


def hbm_roofline(bytes_per_step: float, ms: float, kernel: str) -> dict:
    peak, kind = peaks()
    gbs = bytes_per_step / (ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak, "traffic": None,
            "kernel": kernel, "note": f"peak = {kind} HBM copy bandwidth"}


WORKLOADS = {}


def _contexts(base, adapters, scales, copies, arena_mb, mode=None):
    """`copies` contexts over identical device copies of the base, each with
    `adapters` staged and activated with `scales` (rotated per step so no step
    is L2-resident)."""
    import quantized_base_lora_gb300 as q
    from quantized_base_lora_gb300.runtime import Runtime
    tt = [(t.layer, t.proj, t.d_out, t.d_in, t.qs_off, t.d_off) for t in base.tensors]
    dg = S.content_digest(base.buf)
    ad_dg = [S.content_digest(ad.payload) for ad in adapters]
    rts = []
    for _ in range(copies):
        rt = Runtime(arena_bytes=arena_mb << 20)
        q.check(rt.load_base(base.quant, tt, base.buf, dg), rt.ctx)
        hs = []
        for ad, d in zip(adapters, ad_dg):
            st, h = rt.stage(ad, d)
            q.check(st, rt.ctx)
            hs.append(h)
        if hs:
            q.check(rt.activate(hs, scales, mode if mode is not None else q.OVL_MODE_STACK)[0], rt.ctx)
        rts.append(rt)
    return rts


def _block_step(base, rts, xs, ys, T, sh):
    """One decode step of the block: q+k+v, o, gate+up, down (4 launches)."""
    import quantized_base_lora_gb300 as q
    groups = [[0, 1, 2], [3], [4, 5], [6]]

    def step(i):
        rt = rts[i % len(rts)]
        for grp in groups:
            xp = xs[base.tensors[grp[0]].d_in]
            if len(grp) == 1:
                st = q.ovl_linear_forward(rt.ctx, grp[0], xp, q.OVL_BF16, T, ys[grp[0]], q.OVL_PATH_DUAL, 0, 0, sh)
            else:
                st = q.ovl_linear_forward_multi(rt.ctx, grp, xp, q.OVL_BF16, T, [ys[j] for j in grp], sh)
            if st != 0:
                raise q.OvlError(st, q.ovl_last_error(rt.ctx))
    return step


def _check_all(rts, sh):
    import quantized_base_lora_gb300 as q
    for rt in rts:
        q.check(q.ovl_check_device(rt.ctx, sh), rt.ctx)


def workload_decode_block(args):
    """The headline decode step alone (the 8B-shape q8_0 block + rank-16 LoRA,
    three base copies rotated, activations device-resident): no 32-layer,
    end-to-end or CPU legs.  Small enough to run under a profiler."""
    import torch
    import quantized_base_lora_gb300 as q
    base = S.block_base(S.Q8_0)
    ad = S.block_adapter(base, adapter=0, rank=RANK)
    rts = _contexts(base, [ad], [SCALE], N_COPIES, 64)
    stream = torch.cuda.Stream()
    sh = int(stream.cuda_stream)
    xs = {d: torch.from_numpy(S.to_bf16_bits(S.activations(1, d)).view(np.int16)).cuda().view(torch.bfloat16)
          for d in (4096, 14336)}
    ys = [torch.empty((1, t.d_out), dtype=torch.float32, device="cuda") for t in base.tensors]
    step = block_step(q, base.tensors, sh)
    x_addr = {d: v.data_ptr() for d, v in xs.items()}
    y_ptr = [y.data_ptr() for y in ys]
    ms = timed_steps(lambda i: step(rts[i % N_COPIES], x_addr, y_ptr), args.steps, args.warmup, stream)
    _check_all(rts, sh)
    alg = algorithmic_bytes(base, ad)
    emit({"workload": "decode-block", "metric": METRIC, "unit": "GB/s",
          "value": effective_bytes(base, ad) / (ms / 1e3) / 1e9, "ms_per_step": ms, "steps": args.steps,
          "roofline": hbm_roofline(alg, ms, "k_dualpath (4 launches per step)"),
          "config": {"workload": WORKLOAD, "l2": f"{N_COPIES} base copies rotated"}})


WORKLOADS["decode-block"] = workload_decode_block


def workload_q4_stacked(args):
    import torch
    base = S.block_base(S.Q4_0)
    ads = [S.block_adapter(base, adapter=0, rank=16), S.block_adapter(base, adapter=1, rank=64)]
    rts = _contexts(base, ads, [1.0, 0.5], N_COPIES, 96)
    stream = torch.cuda.Stream()
    sh = int(stream.cuda_stream)
    planes = sum(S.qs_bytes(base.quant, t.d_out, t.d_in) + S.d_bytes(t.d_out, t.d_in) for t in base.tensors)
    lora = sum((16 + 64) * (t.d_in + t.d_out) * 4 for t in base.tensors)
    per_T = {}
    for T in (1, 4, 8):
        xs = {d: torch.from_numpy(S.to_bf16_bits(S.activations(T, d)).view(np.int16)).cuda().view(torch.bfloat16)
              for d in (4096, 14336)}
        ybufs = [torch.empty((T, t.d_out), dtype=torch.float32, device="cuda") for t in base.tensors]
        step = _block_step(base, rts, {d: v.data_ptr() for d, v in xs.items()}, [y.data_ptr() for y in ybufs], T, sh)
        ms = timed_steps(step, args.steps, args.warmup, stream)
        _check_all(rts, sh)
        alg = planes + lora + sum(T * (t.d_in * 2 + t.d_out * 4) for t in base.tensors)
        per_T[T] = {"ms_per_step": ms, "effective_gbs": (planes + lora) / (ms / 1e3) / 1e9,
                    "tok_s": T / (ms / 1e3), "roofline": hbm_roofline(alg, ms, "k_dualpath (4 launches per step)")}
    emit({"workload": "q4-stacked", "metric": "decode effective weight GB/s (8B shape, q4_0 + stacked r16/r64)",
          "unit": "GB/s", "value": per_T[1]["effective_gbs"], "per_T": per_T, "steps": args.steps,
          "config": {"base": "8B-shape block q4_0 (122.7 MB)", "adapters": "r16 s=1.0 then r64 s=0.5 on all 7",
                     "x": "bf16", "l2": f"{N_COPIES} base copies rotated"}})


WORKLOADS["q4-stacked"] = workload_q4_stacked


def workload_q4k_decode(args):
    """The 8B-shape block with a q4_K base (256-weight super-blocks, 4.5 bits per
    weight) and one rank-16 adapter (s = 2.0) on all 7 projections, batch-1
    decode, x bf16: the same step as the headline decode line, q4_K bytes."""
    import torch
    base = S.block_base(S.Q4_K)
    ad = S.block_adapter(base, adapter=0, rank=RANK)
    rts = _contexts(base, [ad], [2.0], N_COPIES, 96)
    stream = torch.cuda.Stream()
    sh = int(stream.cuda_stream)
    planes = sum(S.qs_bytes(base.quant, t.d_out, t.d_in) + S.d_bytes(t.d_out, t.d_in) for t in base.tensors)
    lora = sum(RANK * (t.d_in + t.d_out) * 4 for t in base.tensors)
    per_T = {}
    for T in (1, 64):
        xs = {d: torch.from_numpy(S.to_bf16_bits(S.activations(T, d)).view(np.int16)).cuda().view(torch.bfloat16)
              for d in (4096, 14336)}
        ybufs = [torch.empty((T, t.d_out), dtype=torch.float32, device="cuda") for t in base.tensors]
        step = _block_step(base, rts, {d: v.data_ptr() for d, v in xs.items()}, [y.data_ptr() for y in ybufs], T,
                           sh)
        ms = timed_steps(step, args.steps, args.warmup, stream)
        _check_all(rts, sh)
        alg = planes + lora + sum(T * (t.d_in * 2 + t.d_out * 4) for t in base.tensors)
        if T == 1:
            roof = hbm_roofline(alg, ms, "k_dualpath (4 launches per step)")
        else:
            flops = sum(2 * T * t.d_out * t.d_in for t in base.tensors)
            tf = flops / (ms / 1e3) / 1e12
            roof = {"bound": "tensor", "achieved": tf, "peak": tf32_peak()[0], "unit": "TFLOP/s",
                    "frac": tf / tf32_peak()[0], "traffic": None,
                    "kernel": "k_widen_shrink + k_fused_gemm per group of tensors that share x",
                    "note": f"peak = {tf32_peak()[1]}"}
        per_T[T] = {"ms_per_step": ms, "effective_gbs": (planes + lora) / (ms / 1e3) / 1e9, "tok_s": T * 1e3 / ms,
                    "roofline": roof}
    one = per_T[1]
    emit({"workload": "q4k-decode", "metric": "decode effective weight GB/s & tok/s (8B shape, q4_K + r16 LoRA)",
          "unit": "GB/s", "value": one["effective_gbs"], "ms_per_step": one["ms_per_step"], "tok_s": one["tok_s"],
          "steps": args.steps, "roofline": one["roofline"], "per_T": per_T,
          "config": {"base": f"8B-shape block q4_K ({planes / 1e6:.1f} MB)", "adapter": "r16 s=2.0 on all 7",
                     "x": "bf16", "tokens": "1 (K1) and 64 (tensor-core route)",
                     "l2": f"{N_COPIES} base copies rotated"}})


WORKLOADS["q4k-decode"] = workload_q4k_decode


def workload_sparse_decode(args):
    """The headline decode step (8B-shape q8_0 block, rank-16 LoRA s = 2.0 on all
    7 projections, T = 1, x bf16) with a DARE-style sparse overlay stacked after
    the LoRA on all 7 (1 % of the weights, f16 values, s = 1.0): four k_dualpath
    launches, each followed by one k_sparse_apply over the same tensors."""
    import torch
    import quantized_base_lora_gb300 as q
    from quantized_base_lora_gb300.runtime import Runtime
    base = S.block_base(S.Q8_0)
    ad = S.block_adapter(base, adapter=0, rank=RANK)
    sp = S.block_sparse_adapter(base, adapter=0, keep=0.01)
    tt = [(t.layer, t.proj, t.d_out, t.d_in, t.qs_off, t.d_off) for t in base.tensors]
    dg, ad_dg, sp_dg = S.content_digest(base.buf), S.content_digest(ad.payload), S.content_digest(sp.payload)
    rts = []
    for _ in range(N_COPIES):
        rt = Runtime(arena_bytes=128 << 20)
        q.check(rt.load_base(base.quant, tt, base.buf, dg), rt.ctx)
        st, ha = rt.stage(ad, ad_dg)
        q.check(st, rt.ctx)
        st, hs = rt.stage_sparse(sp, sp_dg)
        q.check(st, rt.ctx)
        q.check(rt.activate([ha, hs], [SCALE, 1.0])[0], rt.ctx)
        rts.append(rt)
    stream = torch.cuda.Stream()
    sh = int(stream.cuda_stream)
    xs = {d: torch.from_numpy(S.to_bf16_bits(S.activations(1, d)).view(np.int16)).cuda().view(torch.bfloat16)
          for d in (4096, 14336)}
    ybufs = [torch.empty((1, t.d_out), dtype=torch.float32, device="cuda") for t in base.tensors]
    step = _block_step(base, rts, {d: v.data_ptr() for d, v in xs.items()}, [y.data_ptr() for y in ybufs], 1, sh)
    ms = timed_steps(step, args.steps, args.warmup, stream)
    _check_all(rts, sh)
    nnz = sum(sp.nnz)
    sparse_bytes = nnz * 6 + sum((t.d_out + 1) * 4 for t in base.tensors)
    eff = effective_bytes(base, ad) + sparse_bytes
    # the sparse pass also reads and rewrites y
    alg = algorithmic_bytes(base, ad) + sparse_bytes + sum(8 * t.d_out for t in base.tensors)
    emit({"workload": "sparse-decode",
          "metric": "decode effective weight GB/s & tok/s (8B shape, q8_0 + r16 LoRA + 1% sparse overlay)",
          "unit": "GB/s", "value": eff / (ms / 1e3) / 1e9, "ms_per_step": ms, "tok_s": 1e3 / ms,
          "steps": args.steps, "nnz": nnz,
          "roofline": hbm_roofline(alg, ms, "k_dualpath (4 launches) + k_sparse_apply (4 launches) per step"),
          "config": {"base": "8B-shape block q8_0", "adapters": "r16 s=2.0 then DARE 1% sparse s=1.0 on all 7",
                     "x": "bf16", "l2": f"{N_COPIES} base copies rotated"}})
    for rt in rts:
        rt.close()


WORKLOADS["sparse-decode"] = workload_sparse_decode


def workload_segmented(args):
    import torch
    import quantized_base_lora_gb300 as q
    base = S.block_base(S.Q4_0, projs=("q", "gate"))
    ads = [S.block_adapter(base, adapter=a, rank=16) for a in range(16)]
    rts = _contexts(base, ads, [2.0] * 16, N_COPIES, 128, mode=q.OVL_MODE_TABLE)
    stream = torch.cuda.Stream()
    sh = int(stream.cuda_stream)
    T = 64
    ids = S.zipf_ids(T, 16, 1.1)
    perm, offsets, slots = S.segments(ids)
    x = torch.from_numpy(S.to_bf16_bits(S.activations(T, 4096)).view(np.int16)).cuda().view(torch.bfloat16)
    ys = [torch.empty((T, t.d_out), dtype=torch.float32, device="cuda") for t in base.tensors]
    offs, sl, pm = [int(v) for v in offsets], [int(v) for v in slots], [int(v) for v in perm]

    def step(i):
        rt = rts[i % len(rts)]
        for j in range(len(base.tensors)):
            st = q.ovl_segmented_forward(rt.ctx, j, x.data_ptr(), q.OVL_BF16, T, offs, sl, pm, ys[j].data_ptr(), sh)
            if st != 0:
                raise q.OvlError(st, q.ovl_last_error(rt.ctx))
    ms = timed_steps(step, args.steps, args.warmup, stream)
    _check_all(rts, sh)
    planes = sum(S.qs_bytes(base.quant, t.d_out, t.d_in) + S.d_bytes(t.d_out, t.d_in) for t in base.tensors)
    lora = 16 * sum(16 * (t.d_in + t.d_out) * 4 for t in base.tensors)
    alg = planes + lora + sum(T * (t.d_in * 2 + t.d_out * 4) for t in base.tensors)
    flops = sum(2 * T * t.d_out * t.d_in for t in base.tensors)
    emit({"workload": "segmented", "metric": "segmented multi-adapter batch time (64 requests, 16 adapters)",
          "unit": "us", "value": ms * 1e3, "higher_is_better": False, "steps": args.steps,
          "tok_s": T / (ms / 1e3), "effective_gbs": (planes + lora) / (ms / 1e3) / 1e9,
          "distinct_adapters": int(len(set(int(v) for v in ids))), "segments": len(sl),
          "roofline": {"bound": "tensor", "achieved": flops / (ms / 1e3) / 1e12, "peak": tf32_peak()[0],
                       "unit": "TFLOP/s", "frac": flops / (ms / 1e3) / 1e12 / tf32_peak()[0], "traffic": None,
                       "kernel": "k_widen_shrink + k_fused_gemm per tensor (64 tokens, all TABLE slots)",
                       "note": f"peak = {tf32_peak()[1]}"},
          "hbm": hbm_roofline(alg, ms, "k_widen_shrink + k_fused_gemm"),
          "config": {"base": "q4_0 q 4096x4096 + gate 14336x4096 (42.5 MB)", "adapters": "16 x r16, s=2.0, TABLE",
                     "requests": "64, Zipf(1.1) seed 3000", "x": "bf16", "l2": f"{N_COPIES} base copies rotated"}})


WORKLOADS["segmented"] = workload_segmented


def workload_prefill_dual(args):
    """The dual path at T = 64, 256 and 512 tokens (tensor-core route, K4): the
    8B-shape q8_0 block with a rank-16 adapter on all seven projections, the
    same four launches per step as decode.  At T = 512 it is the prefill of
    the per-layer JIT workload without any materialized scratch."""
    import torch
    base = S.block_base(S.Q8_0)
    ads = [S.block_adapter(base, adapter=0, rank=16)]
    rts = _contexts(base, ads, [2.0], N_COPIES, 96)
    stream = torch.cuda.Stream()
    sh = int(stream.cuda_stream)
    planes = sum(S.qs_bytes(base.quant, t.d_out, t.d_in) + S.d_bytes(t.d_out, t.d_in) for t in base.tensors)
    lora = sum(16 * (t.d_in + t.d_out) * 4 for t in base.tensors)
    tpeak, tkind = tf32_peak()
    per_T = {}
    for T in (64, 256, 512):
        xs = {d: torch.from_numpy(S.to_bf16_bits(S.activations(T, d)).view(np.int16)).cuda().view(torch.bfloat16)
              for d in (4096, 14336)}
        ybufs = [torch.empty((T, t.d_out), dtype=torch.float32, device="cuda") for t in base.tensors]
        step = _block_step(base, rts, {d: v.data_ptr() for d, v in xs.items()}, [y.data_ptr() for y in ybufs], T, sh)
        ms = timed_steps(step, args.steps if T < 512 else max(3, min(args.steps, 20)), args.warmup, stream)
        _check_all(rts, sh)
        flops = sum(2 * T * t.d_out * t.d_in for t in base.tensors) + sum(2 * T * 16 * (t.d_in + t.d_out)
                                                                          for t in base.tensors)
        tfs = flops / (ms / 1e3) / 1e12
        per_T[T] = {"ms_per_step": ms, "tok_s": T / (ms / 1e3), "effective_gbs": (planes + lora) / (ms / 1e3) / 1e9,
                    "roofline": {"bound": "tensor", "achieved": tfs, "peak": tpeak, "unit": "TFLOP/s",
                                 "frac": tfs / tpeak, "traffic": None,
                                 "kernel": "k_widen_shrink + k_fused_gemm per tensor and 64-token chunk",
                                 "note": f"peak = {tkind}"}}
    emit({"workload": "prefill-dual", "metric": "dual-path multi-token step (8B shape, q8_0 + r16, tensor cores)",
          "unit": "tok/s", "value": per_T[64]["tok_s"], "per_T": per_T, "steps": args.steps,
          "tf32_cublas_tflops_8192cube": tf32_cublas_tflops(),
          "config": {"base": "8B-shape block q8_0 (231.7 MB)", "adapter": "r16 s=2.0 on all 7", "x": "bf16",
                     "T": [64, 256, 512], "l2": f"{N_COPIES} base copies rotated"}})


WORKLOADS["prefill-dual"] = workload_prefill_dual


def tf32_peak():
    """Dense TF32 tensor peak for the roofline: the measured bf16 GEMM burst peak
    (MEASURED_PEAKS.json) x the nominal dense tf32/bf16 ratio of GB300 (1.1 / 2.25
    PFLOP/s, the profiling recipe's table), as the recipe prescribes for a
    contraction in a dtype the peaks file does not carry."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]) * 1.1 / 2.25, "measured bf16 burst x nominal tf32/bf16 (1.1/2.25)"
    except Exception:
        return 1900.0 * 1.1 / 2.25, "fallback bf16 x nominal tf32/bf16 (1.1/2.25)"


_TF32_MEASURED = {}


def tf32_cublas_tflops(m=8192, n=8192, k=8192):
    """A torch (cuBLAS) TF32 matmul of m x k by k x n on this GPU, best of 5
    after warm-up: context for the derived TF32 peak, not its denominator."""
    if (m, n, k) in _TF32_MEASURED:
        return _TF32_MEASURED[(m, n, k)]
    import torch
    old = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        a = torch.randn(m, k, device="cuda")
        b = torch.randn(k, n, device="cuda")
        for _ in range(3):
            torch.matmul(a, b)
        best = float("inf")
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
    finally:
        torch.backends.cuda.matmul.allow_tf32 = old
    _TF32_MEASURED[(m, n, k)] = 2.0 * m * n * k / (best / 1e3) / 1e12
    return _TF32_MEASURED[(m, n, k)]


def workload_jit_prefill(args):
    import torch
    import quantized_base_lora_gb300 as q
    base = S.block_base(S.Q8_0)
    ad = S.block_adapter(base, adapter=0, rank=RANK)
    rt = _contexts(base, [ad], [SCALE], 1, 64)[0]
    stream = torch.cuda.Stream()
    sh = int(stream.cuda_stream)
    T = 512
    xs = {d: torch.from_numpy(S.to_bf16_bits(S.activations(T, d)).view(np.int16)).cuda().view(torch.bfloat16)
          for d in (4096, 14336)}
    ys = [torch.empty((T, t.d_out), dtype=torch.float32, device="cuda") for t in base.tensors]
    need = max((t.d_out * t.d_in * 4 + 127) // 128 * 128 + T * t.d_in * 4 for t in base.tensors) + 256
    scratch = torch.empty(need, dtype=torch.uint8, device="cuda")
    sp = (scratch.data_ptr() + 127) // 128 * 128
    sb = need - (sp - scratch.data_ptr())

    def step(i):
        for j, t in enumerate(base.tensors):
            st = q.ovl_linear_forward(rt.ctx, j, xs[t.d_in].data_ptr(), q.OVL_BF16, T, ys[j].data_ptr(),
                                      q.OVL_PATH_JIT, sp, sb, sh)
            if st != 0:
                raise q.OvlError(st, q.ovl_last_error(rt.ctx))
    steps = max(3, min(args.steps, 20))
    ms = timed_steps(step, steps, min(args.warmup, 3), stream)
    _check_all([rt], sh)
    w = sum(t.d_out * t.d_in for t in base.tensors)
    planes = sum(S.qs_bytes(base.quant, t.d_out, t.d_in) + S.d_bytes(t.d_out, t.d_in) for t in base.tensors)
    lora = sum(RANK * (t.d_in + t.d_out) * 4 for t in base.tensors)
    io = sum(T * (t.d_in * 2 + t.d_in * 4 * 2 + t.d_out * 4) for t in base.tensors)   # x, widened x w+r, y
    alg_bytes = planes + lora + 2 * 4 * w + io          # S written once and read once
    gemm_flop = sum(2 * T * t.d_out * t.d_in for t in base.tensors)
    merge_flop = sum(2 * RANK * t.d_out * t.d_in for t in base.tensors)
    tpk, tkind = tf32_peak()
    hpk, hkind = peaks()
    t_mem = alg_bytes / (hpk * 1e9) * 1e3
    t_tc = gemm_flop / (tpk * 1e12) * 1e3
    emit({"workload": "jit-prefill", "metric": "per-layer JIT prefill time (8B-shape q8_0 layer + r16, T=512)",
          "unit": "ms", "value": ms, "higher_is_better": False, "steps": steps,
          "tok_s": T / (ms / 1e3), "gemm_tflops": gemm_flop / (ms / 1e3) / 1e12,
          "tf32_cublas_tflops_8192cube": tf32_cublas_tflops(),
          "tf32_cublas_tflops_prefill_shape": tf32_cublas_tflops(512, 14336, 4096),
          "roofline": {"bound": "tensor" if t_tc > t_mem else "hbm",
                       "ideal_ms_hbm": t_mem, "ideal_ms_tensor": t_tc, "frac": max(t_mem, t_tc) / ms,
                       "algorithmic_bytes": alg_bytes, "gemm_flop": gemm_flop, "merge_flop": merge_flop,
                       "hbm_peak_gbs": hpk, "tf32_peak_tflops": tpk, "note": f"{hkind}; {tkind}"},
          "config": {"layer": "q,k,v,o,gate,up,down of the 8B block, q8_0", "adapter": "r16 s=2.0", "T": T,
                     "x": "bf16", "path": "k_materialize -> k_widen -> k_jit_gemm per projection"}})


WORKLOADS["jit-prefill"] = workload_jit_prefill

LAYERS = 32


def load_stack(rt, torch, dev, n_layers=LAYERS):
    """Generate the n-layer stack of the 8B-shape q8_0 block (every layer its
    own seeds) straight into one device buffer and register it as the base of
    `rt` (n_layers x 7 tensors, layer-major)."""
    import quantized_base_lora_gb300 as q
    from synth.stack import LayerStack, layer_stride
    buf = torch.empty(n_layers * layer_stride(S.Q8_0), dtype=torch.uint8, device=dev)

    def sink(layer, off, padded):
        buf[off:off + padded.nbytes].copy_(torch.from_numpy(padded))

    stack = LayerStack(S.Q8_0, n_layers, sink)
    torch.cuda.synchronize()
    tensors = [(t.layer, t.proj, t.d_out, t.d_in, t.qs_off, t.d_off) for t in stack.tensors]
    q.check(q.ovl_load_base(rt.ctx, S.Q8_0, tensors, buf.data_ptr(), buf.numel(), stack.digest,
                            int(torch.cuda.current_stream().cuda_stream)), rt.ctx)
    rt.base, rt.tensors = buf, tensors
    return stack


def workload_decode32(args):
    import torch
    import quantized_base_lora_gb300 as q
    stream = torch.cuda.Stream()
    tok = decode32_tok_s(args, q, torch, torch.device("cuda", 0), stream)
    emit({"workload": "decode32", "metric": "32-layer decode tok/s (8B shape, q8_0 + r16 on all 224 tensors)",
          "unit": "tok/s", "value": tok["tok_s"], "ms_per_token": tok["ms_per_token"], "detail": tok,
          "roofline": tok["roofline"],
          "config": {"base": tok["base"], "adapter": "r16 s=2.0 on all 224 tensors, own seeds per tensor",
                     "x": "bf16, the same activation per d_in for every layer", "l2": "7.4 GB working set"}})


WORKLOADS["decode32"] = workload_decode32


def workload_switch(args):
    """Stage a0..a2 (valid) and a3 (declared digest with its first byte
    flipped: must fail), then 100 ops: op 2i activates a_(i mod 4) (a3:
    re-stage, which must fail again), op 2i+1 rolls back.  Host wall time per
    call (every call returns only when its work is done)."""
    import torch
    import quantized_base_lora_gb300 as q
    from quantized_base_lora_gb300.runtime import Runtime
    from synth.stack import stack_adapter
    rt = Runtime(arena_bytes=768 << 20)
    stack = load_stack(rt, torch, torch.device("cuda", 0))
    ads = [stack_adapter(stack, adapter=a, rank=RANK) for a in range(4)]
    digests = [S.content_digest(ad.payload) for ad in ads]
    bad = bytes([digests[3][0] ^ 0xFF]) + digests[3][1:]
    lat = {"stage": [], "stage_corrupt": [], "activate": [], "rollback": []}
    status = {}
    handles = []
    torch.cuda.synchronize()
    for a in range(4):
        t0 = time.perf_counter()
        st, h = rt.stage(ads[a], digests[a] if a < 3 else bad)
        lat["stage" if a < 3 else "stage_corrupt"].append(time.perf_counter() - t0)
        status[st] = status.get(st, 0) + 1
        handles.append(h)
    for i in range(100):
        if i % 2 == 0:
            a = (i // 2) % 4
            t0 = time.perf_counter()
            if a < 3:
                st = rt.activate([handles[a]], [SCALE])[0]
                lat["activate"].append(time.perf_counter() - t0)
            else:
                st, _ = rt.stage(ads[3], bad)
                lat["stage_corrupt"].append(time.perf_counter() - t0)
        else:
            t0 = time.perf_counter()
            st = rt.rollback()[0]
            lat["rollback"].append(time.perf_counter() - t0)
        status[st] = status.get(st, 0) + 1

    def pct(v, p):
        return float(np.percentile(np.array(v) * 1e6, p)) if v else None
    summary = {k: {"n": len(v), "p50_us": pct(v, 50), "p99_us": pct(v, 99), "max_us": pct(v, 100)}
               for k, v in lat.items()}
    st_counts = {q.STATUS_NAMES.get(k, str(k)): c for k, c in status.items()}
    emit({"workload": "switch", "metric": "adapter activate latency p50 (32-layer, 168 MB adapters)",
          "unit": "us", "value": summary["activate"]["p50_us"], "higher_is_better": False,
          "latency": summary, "op_status_counts": st_counts,
          "stage_bytes": int(ads[0].payload.nbytes),
          "config": {"base": f"{LAYERS} layers of the 8B-shape q8_0 block, every layer its own seeds",
                     "adapters": "4 x r16 on all 224 tensors (own seeds per tensor), a3 declared digest corrupted",
                     "ops": "100: activate a_(i mod 4) / rollback alternately"}})


WORKLOADS["switch"] = workload_switch


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["decode"] + sorted(WORKLOADS), default="decode")
    args = ap.parse_args()
    if args.workload != "decode":
        if args.impl == "reference" or args.gpus != 1:
            print(json.dumps({"workload": args.workload, "unavailable": "measured on one GPU, our path only"}))
            return
        WORKLOADS[args.workload](args)
        return
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
