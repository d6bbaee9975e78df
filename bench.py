"""Benchmark: batch-1 dequantize-and-matvec weight stream on GB300.

Default workload (the line the metric is quoted on): the 27B-shaped ternary
decode stack - 60 layers of a GQA transformer (hidden 5120, 40 query / 8 KV
heads of dim 128, SwiGLU intermediate 25600), every linear map in block-128
absmean ternary with fp16 scales (7.27 GB packed), one bf16 activation vector
per layer (one of width 5120 for q/k/v/o/gate/up and one of width 25600 for
down). A step is one batch-1 pass over all 420 matvecs, issued as one
persistent launch.

Other workloads (--workload) measure the remaining hot-path rows in the same
format: the 4096 x 4096 ternary matrix, the INT4 GQA layer set (M = 1 or 4),
the Cassandra draft (M = 1) and target (M = 5) paths on the 14336 x 4096 MLP
matrix, and the 128-expert ternary MoE (M = 1, 2, 4, 8). Workloads smaller
than L2 rotate over enough copies of the packed weights that every step
streams from HBM.

Printed: one JSON line with the achieved HBM GB/s on the algorithmic bytes
(packed weight bytes + activations + outputs), the roofline of the dominant
kernel against the measured copy bandwidth, an end-to-end figure through host
buffers, clocks sampled during the timed region, and (default workload) the
float64 CPU oracle timed on a bounded sample as the CPU baseline.

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
L2_BYTES = 129 * 2 ** 20
DATA = "synthetic (seeded Student-t(4) std 0.02 weights, N(0,1) bf16 activations)"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def captured_traffic(key: str, scale: float = 1.0):
    """DRAM bytes per launch of the dominant kernel from the committed ncu captures
    (profiles/traffic.json), or None when there is no capture for this workload or the
    kernel's source files have changed since it was taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    entry = json.load(open(p))["workloads"].get(key)
    if entry is None:
        return None
    h = hashlib.sha256()
    for f in entry["sources"]:
        h.update(os.path.basename(f).encode())
        h.update(open(os.path.join(ROOT, f), "rb").read())
    if h.hexdigest() != entry["sources_sha256"]:
        return None
    return entry["bytes"] * scale


def copies_for(nbytes: int) -> int:
    """Rotation depth so consecutive steps never find their weights in L2."""
    return max(1, -(-3 * L2_BYTES // nbytes))


PATH_FLAGS = {"auto": 0, "fma": 1, "mma": 2}   # qmv_desc.flags: QMV_FLAG_PATH_FMA / QMV_FLAG_PATH_MMA
MMA_MIN_M = {"int4": 1, "ternary": 2}          # the library's automatic choice of the tensor-core kernel


LUT_KERNEL = "lut_kernel (byte-lookup tables, fp32)"
LUT4_KERNEL = "lut_kernel<INT4> (byte-lookup tables of column pairs, fp32)"


def matvec_kernel(fmt: str, M: int, path: str, layout: str = "record") -> str:
    """Name of the matvec kernel the library runs for this M, layout and kernel choice."""
    if fmt == "ternary" and layout == "lut":
        return LUT_KERNEL
    mma = path == "mma" or (path == "auto" and M >= MMA_MIN_M[fmt])
    if mma:
        return f"gemv_mma_kernel<{fmt}, n-tiles={1 if M <= 8 else 2}> (mma.sync m16n8k16)"
    return f"gemv_kernel<{fmt}, M={min(M, 8)}> (fp16 FMA)"


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
    """Child process: time the float64 oracle on a bounded sample of the stack (one thread).

    The sample unit is the k and v matrices of one layer (2 x 1024 x 5120 weights):
    the oracle decodes their packed bytes, dequantizes and forms y in float64.
    Weights are generated and packed by the oracle before the clock starts; the child
    then prints "ready" and starts its clock when the parent writes a line to its
    standard input, so that all children run at the same time. QMV_ORACLE_PASSES
    fixes the number of passes; otherwise passes repeat until QMV_ORACLE_SECONDS of
    CPU work have been timed.
    """
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
    print("ready", flush=True)
    sys.stdin.readline()
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
    print(json.dumps({"seconds": el, "passes": done, "bytes": nbytes,
                      "weights": sum(N * K for _, N, K in packed)}), flush=True)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_oracle_sample(passes=0, seconds=10.0, cores=None):
    """The oracle's sample on every host core: one single-threaded child per core, all
    started together; throughput = all children's bytes / the slowest child's time."""
    cores = cores or host_cores()
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               QMV_ORACLE_PASSES=str(passes), QMV_ORACLE_SECONDS=str(seconds))
    kids = [subprocess.Popen([sys.executable, os.path.abspath(__file__), "--oracle-child"], env=env, cwd=ROOT,
                             stdin=subprocess.PIPE, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
            for _ in range(cores)]
    try:
        for k in kids:
            if k.stdout.readline().strip() != "ready":
                raise RuntimeError("oracle sample failed: " + k.stderr.read()[-2000:])
        for k in kids:
            k.stdin.write("go\n")
            k.stdin.flush()
        res = []
        for k in kids:
            out, err = k.communicate()
            if k.returncode:
                raise RuntimeError("oracle sample failed: " + err[-2000:])
            res.append(json.loads(out.strip().splitlines()[-1]))
    finally:
        for k in kids:
            if k.poll() is None:
                k.kill()
                k.wait()
    wall = max(r["seconds"] for r in res)
    total = sum(r["bytes"] * r["passes"] for r in res)
    gbs = total / wall / 1e9
    r0 = res[0]
    per_pass = wall / min(r["passes"] for r in res)
    return {"value": gbs, "unit": UNIT, "cores": cores, "kind": "oracle", "seconds_per_pass": per_pass,
            "sample": f"k and v matrices of one stack layer ({r0['weights'] / 1e6:.1f}M weights, "
                      f"{r0['bytes'] / 1e6:.2f} MB packed) decoded, dequantized and multiplied in float64 NumPy; "
                      f"{cores} single-threaded processes (one per host core) at once, "
                      f"{sum(r['passes'] for r in res)} passes in {wall:.2f} s"}


# ----------------------------------------------------------------------------- workloads

class Workload:
    """One batch of synthetic input resident in HBM; step() launches one pass of the hot path."""
    name = ""
    kernel = ""
    tok_s = False

    def config(self):
        raise NotImplementedError

    def step(self, i, stream):
        raise NotImplementedError

    def bytes(self, i):
        return self.nbytes

    def host_io(self):
        """(device inputs, device outputs) that an end-to-end step copies from / to pinned host memory."""
        raise NotImplementedError

    def traffic(self):
        """Captured DRAM bytes per launch of the dominant kernel (None if not captured or stale)."""
        return None


class Stack(Workload):
    name = "stack"
    kernel = "gemv_kernel<ternary, M=1>"
    tok_s = True

    def __init__(self, q, torch, dev, layers=LAYERS, seed=4, path="auto", layout="lut"):
        from quantized_gemv_unpack_gb300 import synth
        self.kernel = matvec_kernel("ternary", 1, path, layout)
        fmt = q.QMV_TERNARY2_LUT if layout == "lut" else q.QMV_TERNARY2
        gen = synth.torch_generator(seed, dev)
        shapes = synth.gqa_layer_shapes(HIDDEN, NQ, NKV, HD, INTER)
        # all activations in one buffer and all outputs in another, so an end-to-end
        # step is one host-to-device and one device-to-host copy
        self.x_all = torch.empty((layers, HIDDEN + INTER), dtype=torch.bfloat16, device=dev)
        self.y_all = torch.empty(layers * sum(N for _, N, _ in shapes), dtype=torch.float32, device=dev)
        tasks = []
        nbytes = 0
        y_off = 0
        for layer in range(layers):
            x_h = self.x_all[layer, :HIDDEN]
            x_i = self.x_all[layer, HIDDEN:]
            x_h.copy_(synth.activations_bf16_torch(gen, (1, HIDDEN), device=dev)[0])
            x_i.copy_(synth.activations_bf16_torch(gen, (1, INTER), device=dev)[0])
            for _, N, K in shapes:
                d = q.qmv_pack_desc(fmt, N, K)
                d.flags = PATH_FLAGS[path] if layout == "record" else 0
                p = torch.empty(d.total_bytes, dtype=torch.uint8, device=dev)
                w = synth.student_t4_torch(gen, (N, K), device=dev)
                q.qmv_pack_ternary(d, w, p)
                del w
                y = self.y_all[y_off:y_off + N].view(1, N)
                y_off += N
                tasks.append((d, p, (x_i if K == INTER else x_h).view(1, K), y))
                nbytes += N * K // 4 + N * (K // 128) * 2 + N * 4
            nbytes += (HIDDEN + INTER) * 2
        torch.cuda.synchronize()
        self.batch = q.Batch(fmt, tasks, 1)
        self.nbytes = nbytes
        self.layers = layers
        self.path = path
        self.layout = layout

    @staticmethod
    def stack_config(layers, layout="lut"):
        return {"workload": f"27B-shaped ternary decode stack: {layers} layers x {{q,k,v,o,gate,up,down}}, "
                            "hidden 5120, 40/8 heads x 128, SwiGLU 25600, block-128 absmean ternary + fp16 scales, "
                            "batch 1",
                "layout": {"lut": "byte-lookup (QMV_TERNARY2_LUT)", "record": "row-group records (QMV_TERNARY2)"}[layout],
                "layers": layers, "hidden": HIDDEN, "heads": [NQ, NKV, HD], "intermediate": INTER,
                "batch": 1, "matvecs_per_step": 7 * layers, "seed": 4,
                "l2": "inputs larger than L2 (7.27 GB of packed weights per step; no flush needed)"}

    def config(self):
        return self.stack_config(self.layers, self.layout)

    def step(self, i, stream):
        self.batch.run(stream)

    def host_io(self):
        return [self.x_all], [self.y_all]

    def traffic(self):
        # the capture is of 3 layers, scaled to 60 there; traffic grows with the layer count
        key = "stack" if self.layout == "lut" else "stack-record"
        return captured_traffic(key, self.layers / LAYERS) if self.path == "auto" else None


class SparseStack(Workload):
    """The 27B-shaped stack with a seeded 16.5 % of its 16 x 128 tiles zero, in the flagged
    sparse ternary format (about 1.78 bits per weight)."""
    name = "stack-sparse"
    kernel = "sparse_kernel<M=1> (fp16 FMA over stored tiles)"
    tok_s = True
    ZERO = 0.165

    def __init__(self, q, torch, dev, layers=LAYERS, seed=4):
        from quantized_gemv_unpack_gb300 import synth
        gen = synth.torch_generator(seed, dev)
        shapes = synth.gqa_layer_shapes(HIDDEN, NQ, NKV, HD, INTER)
        self.x_all = torch.empty((layers, HIDDEN + INTER), dtype=torch.bfloat16, device=dev)
        self.y_all = torch.empty(layers * sum(N for _, N, _ in shapes), dtype=torch.float32, device=dev)
        tasks, self.bufs = [], []
        nbytes = dense_bytes = 0
        y_off = 0
        for layer in range(layers):
            x_h, x_i = self.x_all[layer, :HIDDEN], self.x_all[layer, HIDDEN:]
            x_h.copy_(synth.activations_bf16_torch(gen, (1, HIDDEN), device=dev)[0])
            x_i.copy_(synth.activations_bf16_torch(gen, (1, INTER), device=dev)[0])
            for _, N, K in shapes:
                w = synth.student_t4_torch(gen, (N, K), device=dev)
                zero = torch.rand((N // 16, K // 128), generator=gen, device=dev) < self.ZERO
                w.view(N // 16, 16, K // 128, 128).mul_((~zero).to(w.dtype)[:, None, :, None])
                dense = q.qmv_pack_desc(q.QMV_TERNARY2, N, K)
                p = torch.empty(dense.total_bytes, dtype=torch.uint8, device=dev)
                q.qmv_pack_ternary(dense, w, p)
                del w
                d, host = q.qmv_sparse_pack_host(dense, p.cpu().numpy())
                del p
                sp = torch.from_numpy(host).to(dev)
                self.bufs.append((d, sp))
                y = self.y_all[y_off:y_off + N].view(1, N)
                y_off += N
                tasks.append((d, sp, (x_i if K == INTER else x_h).view(1, K), y))
                nbytes += d.total_bytes + N * 4
                dense_bytes += dense.bytes[0] + N * (K // 128) * 2
            nbytes += (HIDDEN + INTER) * 2
        torch.cuda.synchronize()
        self.batch = q.Batch(q.QMV_TERNARY2_SPARSE, tasks, 1)
        self.nbytes = nbytes
        self.dense_bytes = dense_bytes
        self.layers = layers

    def config(self):
        c = Stack.stack_config(self.layers)
        c["workload"] = c["workload"].replace("block-128 absmean ternary", "flagged sparse block-128 ternary "
                                              f"({100 * self.ZERO:.1f} % of 16 x 128 tiles zero)")
        c["layout"] = "flagged sparse tiles (QMV_TERNARY2_SPARSE)"
        c["zero_tile_fraction"] = self.ZERO
        c["bits_per_weight"] = 8 * (self.nbytes - self.layers * (HIDDEN + INTER) * 2) / sum(
            N * K for _, N, K in synth_shapes()) / self.layers
        c["dense_ternary_bytes"] = self.dense_bytes
        c["l2"] = "inputs larger than L2 (about 6.1 GB of packed weights per step; no flush needed)"
        return c

    def step(self, i, stream):
        self.batch.run(stream)

    def host_io(self):
        return [self.x_all], [self.y_all]

    def traffic(self):
        # captured on 3 layers; every layer's stored tiles are read once, so traffic grows with the layer count
        return captured_traffic("stack-sparse", self.layers / LAYERS)


def synth_shapes():
    from quantized_gemv_unpack_gb300 import synth
    return synth.gqa_layer_shapes(HIDDEN, NQ, NKV, HD, INTER)



class Ternary4096(Workload):
    name = "ternary-4096"
    kernel = "gemv_kernel<ternary, M=1>"

    def __init__(self, q, torch, dev, M=1, path="auto", layout="record"):
        from quantized_gemv_unpack_gb300 import synth
        self.kernel = matvec_kernel("ternary", M, path, layout)
        gen = synth.torch_generator(0, dev)
        N = K = 4096
        self.d = q.qmv_pack_desc(q.QMV_TERNARY2_LUT if layout == "lut" else q.QMV_TERNARY2, N, K)
        self.d.flags = PATH_FLAGS[path] if layout == "record" else 0
        one = torch.empty(self.d.total_bytes, dtype=torch.uint8, device=dev)
        q.qmv_pack_ternary(self.d, synth.student_t4_torch(gen, (N, K), device=dev), one)
        self.copies = copies_for(self.d.total_bytes)
        self.ps = [one.clone() for _ in range(self.copies)]
        self.x = synth.activations_bf16_torch(gen, (M, K), device=dev)
        self.y = torch.empty((M, N), device=dev)
        self.nbytes = self.d.bytes[0] + N * (K // 128) * 2 + M * K * 2 + M * N * 4
        self.M = M
        self.q = q
        self.path = path
        self.layout = layout

    def config(self):
        return {"workload": f"ternary GEMV 4096 x 4096, block-128 absmean + fp16 scales, M={self.M}", "M": self.M,
                "layout": self.layout, "seed": 0, "l2": f"rotating {self.copies} copies of the packed matrix (>= 3x L2)"}

    def step(self, i, stream):
        self.q.qmv_run_ternary(self.d, self.ps[i % self.copies], self.x, self.y, stream)

    def host_io(self):
        return [self.x], [self.y]

    def traffic(self):
        key = f"ternary-4096 M={self.M}" + (" lut" if self.layout == "lut" else "")
        return captured_traffic(key) if self.path == "auto" else None


class Int4Layer(Workload):
    name = "int4-layer"
    kernel = "gemv_kernel<int4, M>"

    def __init__(self, q, torch, dev, M=1, path="auto", layout="record", layers=1):
        from quantized_gemv_unpack_gb300 import synth
        if layout == "lut" and M != 1:
            raise SystemExit("the INT4 lookup layout serves M = 1")
        self.kernel = LUT4_KERNEL if layout == "lut" else matvec_kernel("int4", M, path)
        fmt = q.QMV_INT4_LUT if layout == "lut" else q.QMV_INT4
        gen = synth.torch_generator(1, dev)
        shapes = synth.gqa_layer_shapes(5120, 40, 8, 128, 13824) * layers
        one = []
        for _, N, K in shapes:
            d = q.qmv_pack_desc(fmt, N, K)
            d.flags = PATH_FLAGS[path] if layout == "record" else 0
            p = torch.empty(d.total_bytes, dtype=torch.uint8, device=dev)
            q.qmv_pack_int4(d, synth.student_t4_torch(gen, (N, K), device=dev), p)
            one.append((d, p, N, K))
        layer_bytes = sum(d.total_bytes for d, _, _, _ in one)
        self.copies = copies_for(layer_bytes)
        self.xs = {K: synth.activations_bf16_torch(gen, (M, K), device=dev) for K in (5120, 13824)}
        self.ys = [torch.empty((M, N), device=dev) for _, _, N, _ in one]
        self.batches = []
        for c in range(self.copies):
            tasks = [(d, p if c == 0 else p.clone(), self.xs[K], y) for (d, p, N, K), y in zip(one, self.ys)]
            self.batches.append(q.Batch(fmt, tasks, M))
        self.nbytes = sum(d.bytes[0] + N * (K // 128) * 2 + M * N * 4 for d, _, N, K in one) + M * (5120 + 13824) * 2
        self.M = M
        self.path = path
        self.layout = layout
        self.layers = layers

    def config(self):
        return {"workload": f"INT4 GQA layer set (hidden 5120, 40/8 heads x 128, SwiGLU 13824), group-128 absmax/7, "
                            f"M={self.M}" + (f", {self.layers} layers" if self.layers > 1 else ""),
                "M": self.M, "seed": 1, "matvecs_per_step": 7 * self.layers,
                "layout": {"lut": "byte-lookup (QMV_INT4_LUT)", "record": "row-group records (QMV_INT4)"}[self.layout],
                "l2": f"rotating {self.copies} copies of the layer (>= 3x L2)"}

    def step(self, i, stream):
        self.batches[i % self.copies].run(stream)

    def host_io(self):
        return list(self.xs.values()), self.ys

    def traffic(self):
        key = f"int4-layer M={self.M}" + (" lut" if self.layout == "lut" else "")
        return captured_traffic(key) if self.path == "auto" and self.layers == 1 else None


class Cassandra(Workload):
    kernel = "cass_kernel"

    def __init__(self, q, torch, dev, target=False, mx=False):
        from quantized_gemv_unpack_gb300 import synth
        g = synth.rng(2)
        N, K = 14336, 4096
        W = synth.to_bf16_bits(synth.student_t4(g, (N, K)))
        X, _ = synth.calibration_bf16(g, 128, K)
        self.d, buf = (q.cass_mx_pack_host if mx else q.cass_pack_host)(W, X)
        self.mx = mx
        if mx:
            self.kernel = "cassmx_kernel"
        one = torch.from_numpy(buf).to(dev)
        self.copies = copies_for(self.d.total_bytes)
        self.ps = [one] + [one.clone() for _ in range(self.copies - 1)]
        self.M = 5 if target else 1
        self.x = torch.from_numpy(synth.activations_bf16(g, (self.M, K)).view("int16")).to(dev).view(torch.bfloat16)
        self.y = torch.empty((self.M, N), device=dev)
        n_spec = 4 if mx else 5
        spec = sum(self.d.bytes[i] for i in range(n_spec))
        verif = sum(self.d.bytes[i] for i in range(n_spec, 7 if not mx else 6))
        self.nbytes = (spec + (verif if target else 0)) + self.M * K * 2 + self.M * N * 4
        self.target = target
        self.fn = q.cass_reconstruct if target else q.cass_decode_draft
        self.name = ("cass-mx-" if mx else "cass-") + ("target" if target else "draft")
        self.dense = N * K * 2
        self.spec_bytes, self.verif_bytes = spec, verif
        self.stats = None if mx else exponent_statistics(W, buf, self.d)

    def config(self):
        if self.mx:
            path = ("target (speculation + verification, MX values)" if self.target else "draft (speculation only)")
            name = "Cassandra-2 (MX shared exponent, groups of 32)"
        else:
            path = "target (speculation + verification, bit-exact rebuild)" if self.target else "draft (speculation only)"
            name = "Cassandra split"
        c = {"workload": f"{name} 14336 x 4096 MLP matrix, {path}, M={self.M}", "M": self.M, "seed": 2,
             "dense_bf16_bytes": self.dense, "speculation_bytes": self.spec_bytes,
             "verification_bytes": self.verif_bytes, "n_symbols": self.d.n_symbols,
             "l2": f"rotating {self.copies} copies of the packed matrix (>= 3x L2)"}
        if self.stats:
            c["kept_exponents"] = self.stats
        return c

    def step(self, i, stream):
        self.fn(self.d, self.ps[i % self.copies], self.x, self.y, None, stream)

    def host_io(self):
        return [self.x], [self.y]

    def traffic(self):
        return captured_traffic(f"{self.name} M={self.M}")


def exponent_statistics(W, buf, d):
    """Entropy and mean unary code length (bits) of the kept exponents of a packed Cassandra
    matrix, next to the figures the "Cassandra" page quotes for trained models (section 3.3).
    Read from the packed bitmap (section 0) and the original bf16 weights."""
    import numpy as np
    N, K = W.shape
    words = np.frombuffer(buf, dtype=np.uint32, count=N * K // 32, offset=int(d.off[0])).reshape(N, K // 32)
    keep = ((words[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).astype(bool).reshape(N, K)
    E = ((W[keep] >> 7) & 0xFF).astype(np.int64)
    counts = np.bincount(E, minlength=256)
    p = counts[counts > 0] / counts.sum()
    order = np.lexsort((np.arange(256), -counts))          # rank: count descending, then exponent
    rank = np.empty(256, np.int64)
    rank[order] = np.arange(256)
    return {"entropy_bits": float(-(p * np.log2(p)).sum()), "mean_unary_bits": float((rank[E] + 1).mean()),
            "distinct": int((counts > 0).sum()), "page_trained_models": {"entropy_bits": [2.58, 2.64],
                                                                         "mean_unary_bits": 2.85}}


class CassSpeculate(Cassandra):
    """One draft-then-verify step on the Cassandra matrix: 4 draft matvecs at M = 1 (speculation
    data only), then one target pass at M = 5 (1 + 4 draft tokens) over both streams."""
    name = "cass-speculate"
    kernel = "cass_kernel (4 draft launches at M = 1 + 1 target launch at M = 5)"
    N_DRAFT = 4

    def __init__(self, q, torch, dev):
        super().__init__(q, torch, dev, target=True)
        self.name = "cass-speculate"
        self.kernel = CassSpeculate.kernel
        N, K = 14336, 4096
        self.yd = torch.empty((self.N_DRAFT, N), device=dev)
        self.nbytes = (self.N_DRAFT * (self.spec_bytes + K * 2 + N * 4)
                       + self.spec_bytes + self.verif_bytes + self.M * (K * 2 + N * 4))
        self.q = q

    def config(self):
        c = super().config()
        c["workload"] = ("Cassandra split 14336 x 4096 MLP matrix, one self-speculative step: 4 draft matvecs "
                         "(M=1, speculation data) then one target verification (M=5, both streams)")
        c["n_draft"] = self.N_DRAFT
        return c

    def step(self, i, stream):
        self.q.cass_speculate_step(self.d, self.ps[i % self.copies], self.x, self.yd, self.y, stream)

    def host_io(self):
        return [self.x], [self.yd, self.y]

    def traffic(self):
        return captured_traffic("cass-speculate M=5")


class KvEncode(Workload):
    """Online KV encoder: one decode step's new K and V for the 27B-shaped stack at batch 128
    (60 layers x 2 x 128 token rows of 8 KV heads x 128 = 1024 values), encoded into the
    Cassandra-1 layout with a fixed exponent codebook."""
    name = "kv-encode"
    kernel = "kv_encode_kernel"

    def __init__(self, q, torch, dev, batch=128):
        import numpy as np
        from quantized_gemv_unpack_gb300 import synth
        gen = synth.torch_generator(5, dev)
        self.T, self.D = LAYERS * 2 * batch, NKV * HD
        v = torch.randn((self.T, self.D), generator=gen, device=dev) * 0.5
        v[:, ::64] *= 20                                            # channel outliers, as keys have
        one = v.to(torch.bfloat16)
        E = ((one[:64].view(torch.int16).to(torch.int32) >> 7) & 0xFF).cpu().numpy()
        counts = np.bincount(E.ravel(), minlength=256)
        present = sorted((e for e in range(256) if counts[e]), key=lambda e: (-counts[e], e))
        self.codebook = np.array(present + [e for e in range(256) if not counts[e]], dtype=np.uint8)
        self.slot = self.D * 3 // 32 // 4 * 4                       # 3 bits per kept value on average
        self.copies = copies_for(self.T * self.D * 2)
        self.xs = [one.view(torch.int16)] + [one.view(torch.int16).clone() for _ in range(self.copies - 1)]
        self.d = q.cass_kv_encode(self.xs[0], self.codebook, self.slot)
        self.out = torch.empty(self.d.total_bytes, dtype=torch.uint8, device=dev)
        self.nbytes = self.T * self.D * 2 + self.d.total_bytes
        self.batch, self.q = batch, q

    def config(self):
        return {"workload": f"online KV-cache encoder (Cassandra-1 layout): one decode step's new K and V of the "
                            f"27B-shaped stack at batch {self.batch}: {self.T} token rows x {self.D} bf16",
                "tokens": self.T, "values_per_token": self.D, "slot_words": self.slot, "seed": 5,
                "encoded_bytes": self.d.total_bytes, "input_bytes": self.T * self.D * 2,
                "l2": f"rotating {self.copies} copies of the input (>= 3x L2)"}

    def step(self, i, stream):
        self.q.cass_kv_encode(self.xs[i % self.copies], self.codebook, self.slot, self.out, stream)

    def host_io(self):
        return [self.xs[0]], [self.out]

    def traffic(self):
        return captured_traffic("kv-encode")



class Moe(Workload):
    name = "moe"
    kernel = "moe_expert_kernel<gate|up> + moe_expert_kernel<down> (one step, timed together)"

    _experts = None   # (layout, buffer) shared by the MoE workloads of one process (seed 3)

    @staticmethod
    def kernel_name(layout):
        return ("lut_kernel<gate|up> + lut_kernel<down> (byte-lookup experts, one step, timed together)"
                if layout == "lut" else None)

    def __init__(self, q, torch, dev, M=1, n_logits=64, layout="lut"):
        from quantized_gemv_unpack_gb300 import synth
        E, H, I, topk = 128, 4096, 2048, 8
        fmt = q.QMV_TERNARY2_LUT if layout == "lut" else q.QMV_TERNARY2
        self.gu = q.qmv_pack_desc(fmt, 2 * I, H)
        self.dn = q.qmv_pack_desc(fmt, H, I)
        self.down_off = self.gu.total_bytes
        self.stride = self.down_off + self.dn.total_bytes
        self.layout = layout
        if self.kernel_name(layout):
            self.kernel = self.kernel_name(layout)
        if Moe._experts is None or Moe._experts[0] != layout:
            gen = synth.torch_generator(3, dev)
            buf = torch.empty(E * self.stride, dtype=torch.uint8, device=dev)
            for e in range(E):
                rec = buf[e * self.stride:(e + 1) * self.stride]
                q.qmv_pack_ternary(self.gu, synth.student_t4_torch(gen, (2 * I, H), device=dev), rec[:self.down_off])
                q.qmv_pack_ternary(self.dn, synth.student_t4_torch(gen, (H, I), device=dev), rec[self.down_off:])
            Moe._experts = (layout, buf)
        self.buf = Moe._experts[1]
        gen = synth.torch_generator(30 + M, dev)
        self.logits = [synth.router_logits_torch(gen, M, E, device=dev) for _ in range(n_logits)]
        self.active = [len(set(torch.topk(lg, topk, dim=1).indices.flatten().tolist())) for lg in self.logits]
        self.x = synth.activations_bf16_torch(gen, (M, H), device=dev)
        self.y = torch.empty((M, H), device=dev)
        self.ws = torch.zeros(q.moe_workspace_size(E, topk, M, H, I), dtype=torch.uint8, device=dev)
        self.per_expert = self.gu.bytes[0] + self.gu.bytes[1] + self.dn.bytes[0] + self.dn.bytes[1]
        self.E, self.H, self.I, self.topk, self.M = E, H, I, topk, M
        self.q = q

    def config(self):
        return {"workload": f"MoE decode, 128 ternary SwiGLU experts (hidden 4096, 2048), top-8 softmax, M={self.M}",
                "M": self.M, "seed": 3, "layout": self.layout, "mean_active_experts": sum(self.active) / len(self.active),
                "l2": f"router logits rotate over {len(self.logits)} draws; experts total "
                      f"{self.E * self.stride / 1e6:.0f} MB (> L2)"}

    def bytes(self, i):
        return self.active[i % len(self.active)] * self.per_expert + self.M * self.H * (2 + 4)

    def step(self, i, stream):
        self.q.moe_qmv_run(self.gu, self.dn, self.buf, self.stride, self.down_off, self.E,
                           self.logits[i % len(self.logits)], self.topk, self.x, self.y, self.ws, stream)

    def host_io(self):
        return [self.x], [self.y]

    def traffic(self):
        # the capture is of the first timed step (logits draw 0): scale to the mean active expert count
        t = captured_traffic(f"moe M={self.M}" + (" lut" if self.layout == "lut" else ""))
        return None if t is None else t * (sum(self.active) / len(self.active)) / self.active[0]


def make_workload(name, q, torch, dev, a):
    if name == "stack":
        return Stack(q, torch, dev, a.layers, path=a.path, layout=a.layout or "lut")
    if name == "stack-sparse":
        return SparseStack(q, torch, dev, a.layers)
    if name == "kv-encode":
        return KvEncode(q, torch, dev)
    if name == "ternary-4096":
        return Ternary4096(q, torch, dev, a.M or 1, path=a.path,
                           layout=(a.layout or "record") if (a.M or 1) == 1 else "record")
    if name == "int4-layer":
        # batch 1: the byte-lookup layout (41.0 against 43.2 us on the tensor-core kernel, graph-replayed);
        # M >= 2: the record layout (the lookup kernel serves M = 1)
        lay = a.layout or ("lut" if (a.M or 1) == 1 and a.path == "auto" else "record")
        return Int4Layer(q, torch, dev, a.M or 1, path=a.path, layout=lay, layers=a.int4_layers)
    if name == "cass-speculate":
        return CassSpeculate(q, torch, dev)
    if name in ("cass-draft", "cass-target", "cass-mx-draft", "cass-mx-target"):
        return Cassandra(q, torch, dev, target=name.endswith("target"), mx="-mx-" in name)
    if name == "moe":
        return Moe(q, torch, dev, a.M or 1, layout=a.layout or "lut")
    raise SystemExit(f"unknown workload {name}")


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(values, dist, device):
    """Elementwise maximum of per-rank timings across the process group (the job is as
    slow as its slowest replica)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_throughput(bytes_per_step_per_rank: float, ms_per_step: float, world: int) -> float:
    """Whole-job GB/s: every rank streams its own replica's bytes in the slowest rank's time."""
    return bytes_per_step_per_rank / (ms_per_step * 1e-3) / 1e9 * world


# ----------------------------------------------------------------------------- timing

def time_steps(wl, steps, warmup, stream, torch, graph=False):
    """Mean device time (ms) of `steps` steps after `warmup` untimed ones, CUDA events on `stream`.
    graph: the steps are captured once into a CUDA graph (on torch's capture stream), which is
    replayed once untimed and then timed, so that the kernels run back to back as in a decode loop
    that replays its step graph; otherwise the steps are launched one by one from the host."""
    for i in range(warmup):
        wl.step(i, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream()
            for i in range(steps):
                wl.step(i, cs)
        g.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        del g
        return e0.elapsed_time(e1) / steps
    e0.record(stream)
    for i in range(steps):
        wl.step(i, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


CONFIGS = [  # (key, workload, M): the other four configurations, each on its own workload
    ("cfg1 ternary 4096x4096 M=1", "ternary-4096", 1),
    ("cfg2 INT4 GQA layer set M=1", "int4-layer", 1),
    ("cfg2 INT4 GQA layer set M=4", "int4-layer", 4),
    ("cfg3 Cassandra draft M=1", "cass-draft", 1),
    ("cfg3 Cassandra target M=5", "cass-target", 5),
    ("cfg3 Cassandra 4 drafts + verify M=5", "cass-speculate", 5),
    ("cfg4 MoE 128 experts top-8 M=1", "moe", 1),
    ("cfg4 MoE 128 experts top-8 M=2", "moe", 2),
    ("cfg4 MoE 128 experts top-8 M=4", "moe", 4),
    ("cfg4 MoE 128 experts top-8 M=8", "moe", 8),
]
NOMINAL_HBM_GBS = 8000.0


def measure_configs(q, torch, dev, stream, steps, warmup, peak):
    """Every other configuration, measured in this process under one clock record: time per step
    (the steps replayed as one CUDA graph; the host-launched time beside it), GB/s on the
    algorithmic bytes, fractions of the measured copy peak and of the nominal 8 TB/s, and the ncu
    DRAM traffic per step where a current capture exists."""
    out = {}
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    for key, name, M in CONFIGS:
        args = argparse.Namespace(M=M, path="auto", layout=None, layers=LAYERS, int4_layers=1)
        wl = make_workload(name, q, torch, dev, args)
        ms_host = time_steps(wl, steps, warmup, stream, torch)
        ms = time_steps(wl, steps, warmup, stream, torch, graph=True)
        nb = sum(wl.bytes(i) for i in range(steps)) / steps
        gbs = nb / (ms * 1e-3) / 1e9
        out[key] = {"us_per_step": ms * 1e3, "us_per_step_host_launched": ms_host * 1e3,
                    "GB_s": gbs, "frac_of_measured_copy": gbs / peak,
                    "frac_of_nominal_8TB_s": gbs / NOMINAL_HBM_GBS, "algorithmic_bytes_per_step": nb,
                    "traffic": wl.traffic(), "kernel": wl.kernel, "workload": wl.config()["workload"]}
        if name.startswith("cass"):
            st = wl.config().get("kept_exponents")
            if st:
                out[key]["kept_exponents"] = st
        del wl
        torch.cuda.empty_cache()
    assert q.qmv_check_status() == 0
    out["clocks"] = clocks.stop()
    out["steps_each"] = steps
    out["timing"] = (f"{steps} steps captured as one CUDA graph and replayed (us_per_step); the same steps "
                     f"launched one by one from the host beside it (us_per_step_host_launched)")
    return out


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="qmv", choices=["qmv", "reference"])
    ap.add_argument("--workload", default="stack",
                    choices=["stack", "stack-sparse", "ternary-4096", "int4-layer", "cass-draft", "cass-target",
                             "cass-mx-draft", "cass-mx-target", "cass-speculate", "kv-encode", "moe"])
    ap.add_argument("--M", type=int, default=0, help="activation rows (int4-layer, ternary-4096, moe)")
    ap.add_argument("--path", default="auto", choices=list(PATH_FLAGS),
                    help="matvec kernel: the library's choice by M, or force fp16-FMA / tensor-core")
    ap.add_argument("--layout", default=None, choices=["lut", "record"],
                    help="ternary and INT4 at M = 1 and MoE experts: byte-lookup layout or row-group records "
                         "(default: lookup for the stack, the INT4 layer set at M = 1 and the MoE experts, records "
                         "for the single 4096 x 4096 matrix, where the record kernel is ahead)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="time the steps as one replayed CUDA graph instead of host launches (not for the "
                         "default line)")
    ap.add_argument("--no-configs", action="store_true",
                    help="default workload only: skip measuring the other configurations in the same run")
    ap.add_argument("--layers", type=int, default=LAYERS, help="stack depth (a smaller case for profiling)")
    ap.add_argument("--int4-layers", type=int, default=1, help="INT4 layer sets per step (int4-layer workload)")
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
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA,
                "config": Stack.stack_config(LAYERS, a.layout or "lut"), "impl": "reference",
                "cpu_baseline": {"kind": "oracle", "cores": base["cores"], "sample": base["sample"], "value": base["value"],
                                 "unit": UNIT},
                "e2e": {"value": base["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    # CPU baseline first: a fresh interpreter (fork+exec) before any CUDA work
    cpu = None
    if rank == 0 and a.workload == "stack" and not a.no_cpu_baseline:
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

    wl = make_workload(a.workload, q, torch, dev, a)
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for i in range(a.warmup):
        wl.step(i, stream)
    assert q.qmv_check_status() == 0
    barrier()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier()
    if a.graph:
        ms = time_steps(wl, a.steps, 0, stream, torch, graph=True)
        barrier()
    else:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(a.steps):
            wl.step(i, stream)
        ev1.record(stream)
        barrier()
        ms = ev0.elapsed_time(ev1) / a.steps
    clk = clocks.stop()
    assert q.qmv_check_status() == 0
    nbytes = sum(wl.bytes(i) for i in range(a.steps)) / a.steps

    # end to end through host buffers: inputs from pinned host memory, outputs back to pinned host memory
    ins, outs = wl.host_io()
    ins_h = [t.cpu().pin_memory() for t in ins]
    outs_h = [torch.empty_like(y, device="cpu").pin_memory() for y in outs]
    h2d = sum(t.numel() * t.element_size() for t in ins_h)
    d2h = sum(t.numel() * t.element_size() for t in outs_h)

    def e2e_step(i):
        for h, d_ in zip(ins_h, ins):
            d_.copy_(h, non_blocking=True)
        wl.step(i, stream)
        for d_, h in zip(outs, outs_h):
            h.copy_(d_, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(3, a.steps // 4)
    e0.record(stream)
    for i in range(n_e2e):
        e2e_step(i)
    e1.record(stream)
    barrier()
    ms_e2e = e0.elapsed_time(e1) / n_e2e
    e2e_bytes = sum(wl.bytes(i) for i in range(n_e2e)) / n_e2e

    if dist is not None:
        ms, ms_e2e = max_over_ranks([ms, ms_e2e], dist, dev)
    if rank != 0:
        dist.destroy_process_group()
        return
    peak, peak_kind = peaks()
    configs = None
    if a.workload == "stack" and not a.no_configs:
        configs = measure_configs(q, torch, dev, stream, steps=20, warmup=3, peak=peak)
    per_gpu = job_throughput(nbytes, ms, 1)
    fma_split = 1 if ((a.M or 1) <= 8 or "mma" in wl.kernel) else 2   # fp16-FMA launches cover 8 rows each
    launches = {"stack": 1, "stack-sparse": 1, "ternary-4096": fma_split, "int4-layer": fma_split, "cass-draft": 1,
                "cass-target": 1, "cass-mx-draft": 1, "cass-mx-target": 1, "cass-speculate": 5, "kv-encode": 1,
                "moe": 2}[a.workload]
    line = {
        "metric": METRIC, "value": per_gpu * world, "unit": UNIT, "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if "lut_kernel" in wl.kernel else (
            "fp16x2-f32" if a.workload in ("stack", "stack-sparse", "ternary-4096", "int4-layer", "moe") else "f32"),
        "data": DATA,
        "config": dict(wl.config(), parallelism="replicas only" if world > 1 else "single GPU", kernel_choice=a.path,
                       timing="steps captured as one CUDA graph and replayed" if a.graph else
                       "steps launched one by one from the host"),
        "pct_of_peak": 100.0 * per_gpu / peak,
        "algorithmic_bytes_per_step": nbytes,
        "roofline": {"bound": "hbm", "achieved": per_gpu, "peak": peak, "unit": "GB/s", "frac": per_gpu / peak,
                     "traffic": wl.traffic(), "kernel": wl.kernel, "peak_kind": f"copy bandwidth, {peak_kind}"},
        "e2e": {"value": e2e_bytes / (ms_e2e * 1e-3) / 1e9 * world, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e},
        "gpu_launches": launches * a.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    if configs is not None:
        line["configs"] = configs
    if wl.tok_s:
        line["tok_s"] = 1000.0 / ms * world
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
