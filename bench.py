"""Benchmark: batch-1 dequantize-and-matvec weight stream on GB300.

Default workload: the 27B-shaped ternary decode stack - 60 layers of a GQA
transformer (hidden 5120, 40 query / 8 KV heads of dim 128, SwiGLU
intermediate 25600), every linear map in block-128 absmean ternary with fp16
scales (7.27 GB packed), one bf16 activation vector per layer (one of width
5120 for q/k/v/o/gate/up and one of width 25600 for down). A step is one
batch-1 pass over all 420 matvecs, issued as one persistent launch.

Printed: one JSON line with the achieved HBM GB/s on the algorithmic bytes
(packed codes + scales + activations + outputs), the equivalent decode
tokens/s, the roofline of the dominant kernel against the measured copy
bandwidth, an end-to-end figure through host buffers, and the float64 CPU
oracle timed on a bounded sample as the CPU baseline.

--impl reference times that oracle alone on the host cores (the reference arm).
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
sys.path.insert(0, ROOT)

METRIC = "batch-1 dequant-GEMV achieved HBM GB/s (% of GB300 peak); equiv. decode tok/s"
UNIT = "GB/s"
HIDDEN, NQ, NKV, HD, INTER, LAYERS = 5120, 40, 8, 128, 25600, 60
FALLBACK_HBM_GBS = 6800.0


def workload_config():
    return {"workload": "27B-shaped ternary decode stack: 60 layers x {q,k,v,o,gate,up,down}, hidden 5120, "
                        "40/8 heads x 128, SwiGLU 25600, block-128 absmean ternary + fp16 scales, batch 1",
            "layers": LAYERS, "hidden": HIDDEN, "heads": [NQ, NKV, HD], "intermediate": INTER,
            "batch": 1, "matvecs_per_step": 7 * LAYERS,
            "l2": "inputs larger than L2 (7.27 GB of packed weights per step; no flush needed)",
            "seed": 4}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.out = os.path.join("/tmp", f"qmv_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.out, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.out):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.out)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle sample

def oracle_sample_main():
    """Child process: time the float64 oracle on a bounded sample of the stack (single thread).

    The sample unit is the k and v matrices of one layer (2 x 1024 x 5120 weights):
    the oracle decodes their packed bytes, dequantizes and forms y in float64.
    Weights are generated and packed by the oracle before the clock starts.
    QMV_ORACLE_PASSES fixes the number of passes; otherwise passes repeat until
    QMV_ORACLE_SECONDS of CPU work have been timed.
    """
    import numpy as np

    from oracle import matvec as o_mv
    from oracle import ternary as o_t
    from quantized_gemv_unpack_gb300 import synth
    passes = int(os.environ.get("QMV_ORACLE_PASSES", "0"))
    budget = float(os.environ.get("QMV_ORACLE_SECONDS", "10"))
    g = synth.rng(4)
    shapes = synth.gqa_layer_shapes(HIDDEN, NQ, NKV, HD, INTER)[1:3]
    packed = []
    for _, N, K in shapes:
        w = synth.student_t4(g, (N, K))
        qq, _, s16 = o_t.quantize(w)
        packed.append((o_t.pack(qq, s16), N, K))
    x = synth.activations_bf16(g, (1, HIDDEN))
    nbytes = sum(len(b) for b, _, _ in packed) + HIDDEN * 2 + sum(N for _, N, _ in packed) * 4
    done = 0
    t0 = time.perf_counter()
    while True:
        for buf, N, K in packed:
            qq, s16 = o_t.unpack(buf, N, K)
            o_mv.matvec_bf16x(o_t.dequant(qq, s16), x)
        done += 1
        el = time.perf_counter() - t0
        if (passes and done >= passes) or (not passes and el >= budget):
            break
    print(json.dumps({"seconds": el / done, "passes": done, "bytes": nbytes,
                      "weights": sum(N * K for _, N, K in packed)}))


def run_oracle_sample(passes=0, seconds=10.0):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               QMV_ORACLE_PASSES=str(passes), QMV_ORACLE_SECONDS=str(seconds))
    p = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child"], env=env,
                       capture_output=True, text=True, cwd=ROOT)
    if p.returncode:
        raise RuntimeError("oracle sample failed: " + p.stderr[-2000:])
    r = json.loads(p.stdout.strip().splitlines()[-1])
    gbs = r["bytes"] / r["seconds"] / 1e9
    return {"value": gbs, "unit": UNIT, "cores": 1, "kind": "oracle", "seconds_per_pass": r["seconds"],
            "sample": f"k and v matrices of one stack layer ({r['weights'] / 1e6:.1f}M weights, "
                      f"{r['bytes'] / 1e6:.2f} MB packed) decoded, dequantized and multiplied in float64 NumPy "
                      f"on one thread; {r['passes']} passes, {r['seconds']:.3f} s each"}


# ----------------------------------------------------------------------------- GPU stack

def build_stack(q, torch, dev, layers=LAYERS, seed=4):
    from quantized_gemv_unpack_gb300 import synth
    gen = synth.torch_generator(seed, dev)
    shapes = synth.gqa_layer_shapes(HIDDEN, NQ, NKV, HD, INTER)
    tasks, keep = [], []
    nbytes = 0
    for layer in range(layers):
        x_h = synth.activations_bf16_torch(gen, (1, HIDDEN), device=dev)
        x_i = synth.activations_bf16_torch(gen, (1, INTER), device=dev)
        for name, N, K in shapes:
            d = q.qmv_pack_desc(q.QMV_TERNARY2, N, K)
            p = torch.empty(d.total_bytes, dtype=torch.uint8, device=dev)
            w = synth.student_t4_torch(gen, (N, K), device=dev)
            q.qmv_pack_ternary(d, w, p)
            del w
            y = torch.empty((1, N), dtype=torch.float32, device=dev)
            x = x_i if K == INTER else x_h
            tasks.append((d, p, x, y))
            nbytes += d.bytes[0] + d.bytes[1] + N * 4
        nbytes += (HIDDEN + INTER) * 2
        keep.append((x_h, x_i))
    torch.cuda.synchronize()
    return tasks, keep, nbytes


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="qmv", choices=["qmv", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=LAYERS, help="stack depth (a smaller case for profiling)")
    ap.add_argument("--oracle-child", action="store_true", help=argparse.SUPPRESS)
    a = ap.parse_args()
    if a.oracle_child:
        oracle_sample_main()
        return
    assert a.warmup >= 3, "at least 3 warm-up steps"

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if a.impl == "reference":
        if rank != 0:
            return
        # each step is one oracle pass over its bounded sample of the stack (warm-up passes untimed)
        run_oracle_sample(passes=a.warmup)
        base = run_oracle_sample(passes=a.steps)
        line = {"metric": METRIC, "value": base["value"], "unit": UNIT, "n_gpus": a.gpus, "steps": a.steps,
                "warmup": a.warmup, "ms_per_step": base["seconds_per_pass"] * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded Student-t(4) std 0.02 weights, N(0,1) bf16 activations)",
                "config": workload_config(), "impl": "reference",
                "cpu_baseline": {"kind": "oracle", "cores": 1, "sample": base["sample"], "value": base["value"],
                                 "unit": UNIT},
                "e2e": {"value": base["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    # CPU baseline first: a fresh interpreter (fork+exec) before any CUDA work
    cpu = None
    if rank == 0 and not a.no_cpu_baseline:
        cpu = run_oracle_sample()

    import torch
    import quantized_gemv_unpack_gb300 as q
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    tasks, keep, nbytes = build_stack(q, torch, dev, a.layers)
    batch = q.Batch(q.QMV_TERNARY2, tasks, 1)
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(a.warmup):
        batch.run(stream)
    assert q.qmv_check_status() == 0
    barrier()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(a.steps):
        batch.run(stream)
    ev1.record(stream)
    barrier()
    ms = ev0.elapsed_time(ev1) / a.steps
    clk = clocks.stop()
    launches = a.steps

    # end to end through host buffers: x from pinned host memory in, y back to pinned host memory
    xs_dev = [t for pair in keep for t in pair]
    xs_host = [t.cpu().pin_memory() for t in xs_dev]
    ys_dev = [t[3] for t in tasks]
    ys_host = [torch.empty_like(y, device="cpu").pin_memory() for y in ys_dev]
    h2d = sum(t.numel() * t.element_size() for t in xs_host)
    d2h = sum(t.numel() * t.element_size() for t in ys_host)

    def e2e_step():
        for h, d_ in zip(xs_host, xs_dev):
            d_.copy_(h, non_blocking=True)
        batch.run(stream)
        for d_, h in zip(ys_dev, ys_host):
            h.copy_(d_, non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(3, a.steps // 4)
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e1.record(stream)
    barrier()
    ms_e2e = e0.elapsed_time(e1) / n_e2e

    if dist is not None:
        t = torch.tensor([ms, ms_e2e], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms, ms_e2e = float(t[0]), float(t[1])
    if rank != 0:
        dist.destroy_process_group()
        return
    gbs = nbytes * world / (ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    per_launch_gbs = nbytes / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": gbs, "unit": UNIT, "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp16x2-f32",
        "data": "synthetic (seeded Student-t(4) std 0.02 weights, N(0,1) bf16 activations)",
        "config": dict(workload_config(), layers=a.layers,
                       parallelism="replicas only" if world > 1 else "single GPU"),
        "tok_s": 1000.0 / ms * world, "pct_of_peak": 100.0 * per_launch_gbs / peak,
        "algorithmic_bytes_per_step": nbytes,
        "roofline": {"bound": "hbm", "achieved": per_launch_gbs, "peak": peak, "unit": "GB/s",
                     "frac": per_launch_gbs / peak, "traffic": None,
                     "kernel": "gemv_kernel<ternary, M=1>", "peak_kind": f"copy bandwidth, {peak_kind}"},
        "e2e": {"value": nbytes * world / (ms_e2e * 1e-3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e},
        "gpu_launches": launches,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
