"""Benchmark of the fused dequant-GEMV hot path on one Llama-7B-shaped decoder
layer at decode batch 1 (q/k/v/o 4096x4096 Q4_K, gate/up 11008x4096 Q4_K,
down 4096x11008 Q6_K; x fp32 ~ N(0, 1)).

One step = the seven GEMVs of one layer through the C ABI, i.e. one pass of
the whole hot path: load packed blocks, unpack scales and codes, dequantize
inside the dot product, accumulate, reduce.  Matrices that read the same
activation vector go in one launch, as in a decoder layer: q/k/v
(qk_gemv_batch), o (qk_gemv), gate/up (qk_gemv_batch), down (qk_gemv).  The
step cycles through distinct copies of the layer whose total exceeds the L2
cache, so every step streams its weights from HBM.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on
the host cores instead (a bounded sample of the same workload).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "Q4_K/Q6_K dequant-GEMV HBM GB/s (% of peak); dequant-GEMM TFLOP/s"
L2_BYTES = 129 * 2 ** 20


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def group_bytes(layer, group):
    """Algorithmic bytes of one launch: the group's packed weights, its one
    fp32 activation vector and its fp32 outputs."""
    import synth
    tot = 4 * layer[group[0]][3]
    for i in group:
        (_, name, rows, cols) = layer[i]
        tot += rows * synth.row_bytes(name, cols) + 4 * rows
    return tot


def layer_bytes(layer, groups):
    return sum(group_bytes(layer, g) for g in groups)


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemv_decode_q4k_traffic.json")
KERNEL_SOURCES = ["qk_hgemv.cu", "qk_hunits.cuh", "qk_ptx.cuh", "qk_formats.cuh"]


def kernel_sources_digest():
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "gguf_quant_dequant_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(key="mean_dram_bytes_per_launch"):
    """DRAM bytes per decode launch from the committed ncu summary: the mean
    over the Q4_K launches of the step (q/k/v, o, gate/up), or with
    key="q6k_dram_bytes_per_launch" the Q6_K down launch; None when the
    kernel sources changed since it was captured."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
        if rec.get("kernel_sources_sha256") != kernel_sources_digest():
            return None
        return float(rec[key])
    except Exception:
        return None


# 4 launches per step (q/k/v, o, gate/up, down); skip 8 warm-up steps, take 3.
TRAFFIC_COMMAND = ("ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum "
                   "--clock-control none -k regex:hgemv -s 32 -c 12 --csv --log-file traffic.csv "
                   "python bench.py --steps 20 --warmup 3 --min-warmup-s 0 --no-cpu --no-gemm --no-stack "
                   "--no-sweep --no-quant --no-swiglu --no-attn --no-codes-check")


def record_traffic(csv_path: str) -> dict:
    """Write TRAFFIC_FILE from the launch list of TRAFFIC_COMMAND: DRAM bytes
    (read + write) per decode launch, labelled q/k/v, o, gate/up, down in
    step order, with the digest of the kernel sources it was taken on."""
    import csv
    rows = list(csv.reader(open(csv_path)))
    h = next(i for i, r in enumerate(rows) if "Metric Name" in r)
    hdr, data = rows[h], rows[h + 1:]
    ki, mi, vi, ii = hdr.index("Kernel Name"), hdr.index("Metric Name"), hdr.index("Metric Value"), hdr.index("ID")
    launches = {}
    for r in data:
        if len(r) > vi:
            launches.setdefault(r[ii], {"kernel": r[ki]})[r[mi]] = float(r[vi].replace(",", ""))
    labels = ("qkv", "o", "gate_up", "down")
    per = {lab: [] for lab in labels}
    for n, v in enumerate(launches.values()):
        per[labels[n % 4]].append(v["dram__bytes_read.sum"] + v["dram__bytes_write.sum"])
    means = {lab: int(round(sum(x) / len(x))) for lab, x in per.items() if x}
    q4 = [means[lab] for lab in ("qkv", "o", "gate_up") if lab in means]
    rec = {"kernel": "hgemv_kernel<Q4_K> (q/k/v, o, gate/up) and hgemv_kernel<Q6_K> (down): the tensor-core "
                     "decode GEMV, the four launches of one Llama-7B-shaped layer step",
           "command": TRAFFIC_COMMAND, "dram_bytes_per_launch": means,
           "mean_dram_bytes_per_launch": int(round(sum(q4) / len(q4))),
           "q6k_dram_bytes_per_launch": means.get("down"),
           "note": "read + write; writes are ~0 (the outputs stay in L2 within the launch)",
           "kernel_sources": KERNEL_SOURCES, "kernel_sources_sha256": kernel_sources_digest()}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(rec, f, indent=1)
    return rec


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.f = None

    def __enter__(self):
        try:
            self.f = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.f is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.f.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def build_layer_copies(dev, ncopies, quantized=True):
    """ncopies distinct layers of packed weights on the device, plus one
    activation vector per launch group and one output per matrix.  The codes
    come from the library's quantizer applied to seeded N(0, 0.02) fp32
    weights, or (quantized=False) are seeded random bytes with random fp16
    scales."""
    import torch
    import gguf_quant_dequant_gb300 as qk
    import synth
    layer, groups = synth.LLAMA7B_LAYER, synth.LLAMA7B_LAYER_GROUPS
    Ws = []
    for c in range(ncopies):
        Wc = []
        for i, (_, name, rows, cols) in enumerate(layer):
            if quantized:
                gw = torch.Generator(device=dev)
                gw.manual_seed(100 * c + i)
                w = torch.randn((rows, cols), device=dev, generator=gw) * 0.02
                Wc.append(qk.quantize(synth.TYPE_IDS[name], w))
                del w
            else:
                Wc.append(synth.random_blocks_torch(name, rows, cols, 100 * c + i, dev))
        Ws.append(Wc)
    g = torch.Generator(device=dev)
    g.manual_seed(4242)
    xs = [torch.randn(layer[grp[0]][3], device=dev, generator=g) for grp in groups]
    ys = [torch.empty(rows, device=dev) for (_, _, rows, _) in layer]
    torch.cuda.synchronize()
    return layer, groups, Ws, xs, ys


def run_group(layer, grp, W, x, ys):
    """One launch: qk_gemv for a single matrix, qk_gemv_batch for a group."""
    import gguf_quant_dequant_gb300 as qk
    import synth
    (_, name, rows, cols) = layer[grp[0]]
    t = synth.TYPE_IDS[name]
    if len(grp) == 1:
        qk.gemv(t, W[grp[0]], rows, cols, x.view(1, cols), y=ys[grp[0]].view(1, rows))
    else:
        qk.gemv_batch(t, [W[i] for i in grp], [layer[i][2] for i in grp], cols, x, ys=[ys[i] for i in grp])


def run_gpu(args):
    import torch
    import gguf_quant_dequant_gb300 as qk
    import synth
    from gguf_quant_dequant_gb300 import build as qkbuild

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    qkbuild.build()
    qk.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    hbm_peak, peak_src = peaks()

    wbytes = sum(rows * synth.row_bytes(name, cols) for (_, name, rows, cols) in synth.LLAMA7B_LAYER)
    ncopies = max(2, -(-4 * L2_BYTES // wbytes))
    layer, groups, Ws, xs, ys = build_layer_copies(dev, ncopies)
    lb = layer_bytes(layer, groups)
    for grp in groups:   # every launch runs the decode kernel (no workspace, no prep kernel)
        (_, name, rows, cols) = layer[grp[0]]
        assert qk.gemv_workspace(synth.TYPE_IDS[name], rows, cols, 1) == 0

    def step(c):
        for gi, grp in enumerate(groups):
            run_group(layer, grp, Ws[c], xs[gi], ys)

    def sub_step(c, gidx):
        for gi in gidx:
            run_group(layer, groups[gi], Ws[c], xs[gi], ys)

    # Warm the kernels up eagerly once (module load, attributes), then capture
    # the steps of all layer copies back to back in one CUDA graph (as a
    # model's forward pass over consecutive layers is captured), plus one
    # graph per copy for a remainder of steps.
    for c in range(ncopies):
        step(c)
    torch.cuda.synchronize()

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    q4_groups = [gi for gi, grp in enumerate(groups) if layer[grp[0]][1] == "Q4_K"]
    q6_groups = [gi for gi, grp in enumerate(groups) if layer[grp[0]][1] == "Q6_K"]
    g_all = capture(lambda: [step(c) for c in range(ncopies)])
    graphs = [capture(lambda c=c: step(c)) for c in range(ncopies)]
    q4_all = capture(lambda: [sub_step(c, q4_groups) for c in range(ncopies)])
    q6_all = capture(lambda: [sub_step(c, q6_groups) for c in range(ncopies)])
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def run_steps(n, whole, single):
        for _ in range(n // ncopies):
            whole.replay()
        for k in range(n % ncopies):
            single[k].replay()

    K, W = args.steps, args.warmup
    with Clocks(local) as clk:
        t_end = time.time() + args.min_warmup_s
        i = 0
        while i < W or time.time() < t_end:
            g_all.replay()
            i += ncopies
            if i % (16 * ncopies) == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        _barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_steps(K, g_all, graphs)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        _barrier(world)
        torch.cuda.synchronize()
        # Dominant kernel alone: the three Q4_K launches of a layer (q/k/v,
        # o, gate/up), same rotation.
        reps = max(K // ncopies, 40)
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(reps):
            q4_all.replay()
        f1.record(stream)
        torch.cuda.synchronize()
        q4_ms = f0.elapsed_time(f1)
        # The Q6_K down launch alone, same rotation.
        f0.record(stream)
        for _ in range(reps):
            q6_all.replay()
        f1.record(stream)
        torch.cuda.synchronize()
        q6_ms = f0.elapsed_time(f1)
    clocks = clk.summary()
    ms_max = _max_over_ranks(ms, world)
    ms_step = ms_max / K
    value = world * lb / (ms_step * 1e-3) / 1e9

    q4_launch_bytes = sum(group_bytes(layer, groups[gi]) for gi in q4_groups) / len(q4_groups)
    q4_launch_ms = q4_ms / (reps * ncopies * len(q4_groups))
    achieved = q4_launch_bytes / (q4_launch_ms * 1e-3) / 1e9
    q6_launch_bytes = sum(group_bytes(layer, groups[gi]) for gi in q6_groups) / len(q6_groups)
    q6_launch_ms = q6_ms / (reps * ncopies * len(q6_groups))
    achieved_q6 = q6_launch_bytes / (q6_launch_ms * 1e-3) / 1e9

    # The same step on random-byte codes (random fp16 scales), to show the
    # timing does not depend on how the codes were made.
    codes_check = None
    if not args.no_codes_check:
        del graphs, g_all, q4_all, q6_all
        _, _, Wr, _, _ = build_layer_copies(dev, ncopies, quantized=False)
        gr = capture(lambda: [[run_group(layer, grp, Wr[c], xs[gi], ys) for gi, grp in enumerate(groups)]
                              for c in range(ncopies)])
        for _ in range(3):
            gr.replay()
        torch.cuda.synchronize()
        r0 = torch.cuda.Event(enable_timing=True)
        r1 = torch.cuda.Event(enable_timing=True)
        nrep = max(K // ncopies, 1)
        r0.record(stream)
        for _ in range(nrep):
            gr.replay()
        r1.record(stream)
        torch.cuda.synchronize()
        rand_step = r0.elapsed_time(r1) / (nrep * ncopies)
        codes_check = {"quantized_codes_ms_per_step": round(ms / K, 6),
                       "random_byte_codes_ms_per_step": round(rand_step, 6),
                       "ratio_random_over_quantized": round(rand_step / (ms / K), 4)}
        del Wr, gr
        graphs = g_all = q4_all = q6_all = None

    e2e = run_e2e(args, dev, layer, groups, Ws[0], xs, lb) if rank == 0 else None
    del Ws, graphs, g_all, q4_all, q6_all
    torch.cuda.empty_cache()
    stack = run_stack(dev) if (rank == 0 and not args.no_stack) else None
    sweep = run_ffn_sweep(dev) if (rank == 0 and not args.no_sweep) else None
    gemm = None
    if rank == 0 and not args.no_gemm:
        gemm = run_gemm_bench(dev)
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                pk = json.load(f)
            gemm["frac_of_bf16_peak"] = round(gemm["tflops"] / float(pk["bf16_tflops"]), 4)
            gemm["frac_of_bf16_sustained"] = round(gemm["tflops"] / float(pk["bf16_tflops_sustained"]), 4)
        except Exception:
            pass
    quant = run_quantize(dev, hbm_peak) if (rank == 0 and not args.no_quant) else None
    swi = run_swiglu(dev, hbm_peak) if (rank == 0 and not args.no_swiglu) else None
    attn = run_attn(dev, hbm_peak) if (rank == 0 and not args.no_attn) else None
    cpu = cpu_baseline(layer) if (rank == 0 and world == 1 and not args.no_cpu) else None
    traffic = recorded_traffic()
    if rank == 0:
        out = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": round(ms_step, 6), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "q4_k/q6_k blocks, f32 activations and accumulation",
            "data": "synthetic (codes from qk_quantize of seeded N(0, 0.02) fp32 weights, x ~ N(0,1))",
            "config": {"workload": "Llama-7B-shaped decoder layer, decode batch 1: q/k/v/o 4096x4096 Q4_K, "
                                   "gate/up 11008x4096 Q4_K, down 4096x11008 Q6_K",
                       "launches": "q/k/v one qk_gemv_batch (shared x), o qk_gemv, gate/up one qk_gemv_batch "
                                   "(shared x), down qk_gemv",
                       "bytes_per_step": lb, "layer_copies_rotated": ncopies,
                       "l2": f"inputs larger than L2: {ncopies} distinct layer copies "
                             f"({ncopies * wbytes / 2**20:.0f} MiB) rotated per step",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "timing": f"one CUDA graph of {ncopies} consecutive layer steps (one per copy), "
                                 "replayed; CUDA events on the launch stream"},
            "frac_of_peak": round(value / world / hbm_peak, 4),
            "roofline": {"bound": "hbm", "kernel": "hgemv_kernel<Q4_K> (decode; q/k/v, o and gate/up launches)",
                         "achieved": round(achieved, 2), "peak": hbm_peak, "peak_source": peak_src, "unit": "GB/s",
                         "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                         "launch_bytes": int(q4_launch_bytes), "launch_us": round(q4_launch_ms * 1e3, 3)},
            "roofline_q6k": {"bound": "hbm", "kernel": "hgemv_kernel<Q6_K> (decode; the down launch)",
                             "achieved": round(achieved_q6, 2), "peak": hbm_peak, "peak_source": peak_src,
                             "unit": "GB/s", "frac": round(achieved_q6 / hbm_peak, 4),
                             "traffic": recorded_traffic("q6k_dram_bytes_per_launch"),
                             "launch_bytes": int(q6_launch_bytes), "launch_us": round(q6_launch_ms * 1e3, 3)},
            "codes_check": codes_check,
            "gpu_launches": K * len(groups),
            "clocks": clocks,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gemm": gemm,
            "stack": stack,
            "ffn_sweep": sweep,
            "quantize": quant,
            "swiglu": swi,
            "kv_attention": attn,
        }
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_gemm_bench(dev, reps: int = 5):
    """Prefill dequant-GEMM (M = 2048 bf16 activations) over the mixed recipe
    of 4096x4096, 14336x4096 and 4096x14336 matrices in Q4_K / Q6_K / Q8_0
    plus the 128256x4096 Q6_K vocabulary matrix.  TFLOP/s = 2*M*N*K / time
    (CUDA events, median of `reps` launches per matrix), and the same flops
    through qk_dequant -> bf16 + torch.matmul (cuBLAS) as a comparator."""
    import torch
    import gguf_quant_dequant_gb300 as qk
    import synth
    M = synth.PREFILL_M
    g = torch.Generator(device=dev)
    g.manual_seed(77)
    stream = torch.cuda.current_stream()
    per, tot_flop, tot_ms, cmp_flop, cmp_ms = {}, 0.0, 0.0, 0.0, 0.0
    Xs = {}
    for i, (nm, name, rows, cols) in enumerate(synth.PREFILL):
        t = synth.TYPE_IDS[name]
        W = synth.random_blocks_torch(name, rows, cols, 900 + i, dev)
        if cols not in Xs:
            Xs[cols] = torch.randn((M, cols), device=dev, generator=g).to(torch.bfloat16)
        X = Xs[cols]
        Y = torch.empty((M, rows), device=dev)
        for _ in range(2):
            qk.gemm(t, W, rows, cols, X, Y=Y)
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            qk.gemm(t, W, rows, cols, X, Y=Y)
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        ms = statistics.median(ts)
        fl = 2.0 * M * rows * cols
        per[nm] = round(fl / (ms * 1e-3) / 1e12, 1)
        tot_flop += fl
        tot_ms += ms
        if nm != "vocab":
            Wb = torch.empty((rows, cols), dtype=torch.bfloat16, device=dev)
            for _ in range(2):
                qk.dequant(t, W, rows, cols, out=Wb, bf16=True)
                torch.matmul(X, Wb.t())
            ts = []
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                qk.dequant(t, W, rows, cols, out=Wb, bf16=True)
                torch.matmul(X, Wb.t())
                e1.record(stream)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1))
            cmp_flop += fl
            cmp_ms += statistics.median(ts)
            del Wb
        del W, Y
    torch.cuda.synchronize()
    return {"workload": "prefill dequant-GEMM, M=2048 bf16 activations, 9 recipe matrices + 128256x4096 Q6_K vocab",
            "tflops": round(tot_flop / (tot_ms * 1e-3) / 1e12, 1), "per_matrix_tflops": per,
            "comparator_dequant_then_cublas_tflops": round(cmp_flop / (cmp_ms * 1e-3) / 1e12, 1),
            "comparator_note": "qk_dequant to bf16 then torch.matmul, same 9 matrices (vocab excluded)"}


def run_ffn_gemm(dev, M: int, reps: int = 20):
    """Small-batch dequant-GEMM alone: the Llama-3-8B FFN matrices (gate/up
    14336x4096, down 4096x14336) in Q4_K through qk_gemm at activation batch
    M, four rotating weight copies (beyond L2).  Per matrix: 2 warm-up launches,
    then `reps` launches back to back between two CUDA events; GB/s counts
    packed weights + X (bf16) + Y (fp32)."""
    import torch
    import gguf_quant_dequant_gb300 as qk
    import synth
    t = qk.Q4_K
    stream = torch.cuda.current_stream()
    g = torch.Generator(device=dev)
    g.manual_seed(4242)
    out = {}
    for i, (nm, name, rows, cols) in enumerate(synth.llama3_ffn("Q4_K")):
        Ws = [synth.random_blocks_torch(name, rows, cols, 8000 + 10 * i + k, dev) for k in range(4)]
        X = torch.randn((M, cols), device=dev, generator=g).to(torch.bfloat16)
        Y = torch.empty((M, rows), device=dev)
        ws = torch.empty(max(16, qk.gemm_workspace(t, rows, cols, M)), dtype=torch.uint8, device=dev)
        for k in range(2):
            qk.gemm(t, Ws[k], rows, cols, X, Y=Y, ws=ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k in range(reps):
            qk.gemm(t, Ws[k % 4], rows, cols, X, Y=Y, ws=ws)
        e1.record(stream)
        e1.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        nbytes = Ws[0].numel() + 2 * M * cols + 4 * M * rows
        out[nm] = {"us": round(us, 2), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                   "tflops": round(2.0 * M * rows * cols / (us * 1e-6) / 1e12, 2)}
        del Ws, X, Y, ws
    return {"workload": f"Llama-3-8B FFN Q4_K, qk_gemm at M={M}", "per_matrix": out}


def run_swiglu(dev, hbm_peak=None):
    """Decode SwiGLU gate h = SiLU(Wg x) * (Wu x) in Q4_K for the Llama-7B
    (11008x4096) and Llama-3-8B (14336x4096) FFN: the fused qk_gemv_swiglu
    (one launch, h only) against qk_gemv_batch(gate, up) followed by
    torch's silu(g) * u.  Four weight copies rotate (beyond L2), each timed
    as a CUDA graph.  GB/s counts both matrices' packed bytes + x + h."""
    import torch
    import gguf_quant_dequant_gb300 as qk
    import synth
    t = qk.Q4_K
    out = {}
    for label, rows, cols in (("llama7b_gate_up", 11008, 4096), ("llama3_8b_gate_up", 14336, 4096)):
        nc = 4
        Wg = [synth.random_blocks_torch("Q4_K", rows, cols, 9100 + k, dev) for k in range(nc)]
        Wu = [synth.random_blocks_torch("Q4_K", rows, cols, 9200 + k, dev) for k in range(nc)]
        x = torch.randn(cols, device=dev)
        h = torch.empty(rows, device=dev)
        g = torch.empty(rows, device=dev)
        u = torch.empty(rows, device=dev)

        def fused():
            for k in range(nc):
                qk.gemv_swiglu(t, Wg[k], Wu[k], rows, cols, x, h=h)

        def unfused():
            for k in range(nc):
                qk.gemv_batch(t, [Wg[k], Wu[k]], [rows, rows], cols, x, ys=[g, u])
                torch.mul(torch.nn.functional.silu(g), u, out=h)

        us_f = _graph_time_us(fused) / nc
        us_u = _graph_time_us(unfused) / nc
        nbytes = 2 * Wg[0].numel() + 4 * cols + 4 * rows
        out[label] = {"fused_us": round(us_f, 2), "unfused_us": round(us_u, 2),
                      "fused_gbs": round(nbytes / (us_f * 1e-6) / 1e9, 1),
                      "unfused_gbs": round(nbytes / (us_u * 1e-6) / 1e9, 1)}
        if hbm_peak:
            out[label]["fused_frac_of_hbm"] = round(nbytes / (us_f * 1e-6) / 1e9 / hbm_peak, 4)
        del Wg, Wu
    return {"workload": "decode SwiGLU gate, Q4_K, batch 1", "per_shape": out}


def run_attn(dev, hbm_peak=None):
    """Decode attention over a quantized KV cache (qk_attn_decode): Llama-3-8B
    heads (32 query, 8 kv, d = 128) at 32k positions, one query token, the
    cache in Q8_0 and in Q4_0.  Three cache copies rotate (beyond L2), timed
    as a CUDA graph.  GB/s counts the K and V bytes (the queries and output
    are a few KB)."""
    import torch
    import gguf_quant_dequant_gb300 as qk
    import synth
    Tn, nh, nkv, d = 32768, 32, 8, 128
    out = {}
    for name in ("Q8_0", "Q4_0"):
        t = synth.TYPE_IDS[name]
        nc = 3
        Ks = [synth.random_blocks_torch(name, Tn * nkv, d, 9300 + k, dev) for k in range(nc)]
        Vs = [synth.random_blocks_torch(name, Tn * nkv, d, 9400 + k, dev) for k in range(nc)]
        q = torch.randn((nh, d), device=dev)
        o = torch.empty((nh, d), device=dev)
        ws = torch.empty(qk.attn_decode_workspace(t, Tn, nh, nkv, d), dtype=torch.uint8, device=dev)

        def step():
            for k in range(nc):
                qk.attn_decode(t, q, Ks[k], Vs[k], Tn, nh, nkv, d, 1.0 / d ** 0.5, out=o, ws=ws)

        us = _graph_time_us(step) / nc
        nbytes = 2 * Ks[0].numel()
        out[name] = {"us": round(us, 2), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1), "kv_bytes": nbytes}
        if hbm_peak:
            out[name]["frac_of_hbm"] = round(nbytes / (us * 1e-6) / 1e9 / hbm_peak, 4)
        del Ks, Vs
    return {"workload": "decode attention, 32 query / 8 kv heads, d = 128, 32768 cached positions",
            "per_cache_type": out}


def run_quantize(dev, hbm_peak=None, reps: int = 20, imx_reps: int = 3):
    """The write side: qk_quantize of one 14336x4096 fp32 matrix (N(0, 0.02),
    235 MB, beyond L2) into each block type.  Per type: 2 warm-up launches,
    then `reps` launches back to back between two CUDA events.  GB/s counts
    the 4 bytes read and the packed bytes written per weight.  The
    importance-weighted quantizer (qk_quantize_imatrix, log-normal column
    importances exp(N(0, 1))) is timed the same way with one warm-up and
    `imx_reps` launches: it is bound by its candidate search, so its figure
    is microseconds and weights per second."""
    import torch
    import gguf_quant_dequant_gb300 as qk
    import synth
    rows, cols = 14336, 4096
    stream = torch.cuda.current_stream()
    g = torch.Generator(device=dev)
    g.manual_seed(2024)
    w = torch.randn((rows, cols), device=dev, generator=g) * 0.02
    imp = torch.exp(torch.randn(cols, device=dev, generator=g))
    per = {}
    for name in ("Q4_K", "Q6_K", "Q8_0", "Q5_0", "Q4_0", "Q5_K", "Q2_K", "Q3_K"):
        t = synth.TYPE_IDS[name]
        o = torch.empty(rows * qk.row_bytes(t, cols), dtype=torch.uint8, device=dev)
        for _ in range(2):
            qk.quantize(t, w, out=o)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            qk.quantize(t, w, out=o)
        e1.record(stream)
        e1.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        gbs = (4 * rows * cols + o.numel()) / (us * 1e-6) / 1e9
        per[name] = {"us": round(us, 2), "gbs": round(gbs, 1)}
        if hbm_peak:
            per[name]["frac_of_hbm"] = round(gbs / hbm_peak, 4)
        if imx_reps > 0:
            qk.quantize_imatrix(t, w, imp, out=o)
            e0.record(stream)
            for _ in range(imx_reps):
                qk.quantize_imatrix(t, w, imp, out=o)
            e1.record(stream)
            e1.synchronize()
            ius = e0.elapsed_time(e1) * 1e3 / imx_reps
            per[name]["imatrix_us"] = round(ius, 1)
            per[name]["imatrix_gweights_per_s"] = round(rows * cols / (ius * 1e-6) / 1e9, 2)
        del o
    del w, imp
    return {"workload": "qk_quantize and qk_quantize_imatrix, 14336x4096 fp32 N(0, 0.02) -> each block type",
            "per_type": per}


def _graph_time_us(fn, reps: int = 20, warm: int = 3) -> float:
    """Median over reps of one replay of a CUDA graph of fn, in microseconds."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    del g
    return statistics.median(ts)


def run_stack(dev):
    """The full Llama-7B-shaped stack at decode batch 1 (32 layers in the
    bench's four launches each, lm_head 32000x4096 Q6_K, two 4096^2 Q8_0):
    one token = one pass over 3.87 GiB of packed weights, captured in one
    CUDA graph.  Reports tokens/s-equivalent and GB/s."""
    import torch
    import gguf_quant_dequant_gb300 as qk
    import synth
    layer, groups = synth.LLAMA7B_LAYER, synth.LLAMA7B_LAYER_GROUPS
    g = torch.Generator(device=dev)
    g.manual_seed(5151)
    L = 32
    Ws = [[synth.random_blocks_torch(name, rows, cols, 6000 + 10 * l + i, dev)
           for i, (_, name, rows, cols) in enumerate(layer)] for l in range(L)]
    tail = [("Q6_K", 32000, 4096), ("Q8_0", 4096, 4096), ("Q8_0", 4096, 4096)]
    Wt = [synth.random_blocks_torch(n, r, c, 6900 + i, dev) for i, (n, r, c) in enumerate(tail)]
    xs = [torch.randn(layer[grp[0]][3], device=dev, generator=g) for grp in groups]
    x4 = torch.randn(4096, device=dev, generator=g)
    ys = [torch.empty(rows, device=dev) for (_, _, rows, _) in layer]
    yt = [torch.empty(r, device=dev) for (_, r, _) in tail]
    nbytes = sum(w.numel() for ws_ in Ws for w in ws_) + sum(w.numel() for w in Wt)

    def token():
        for l in range(L):
            for gi, grp in enumerate(groups):
                run_group(layer, grp, Ws[l], xs[gi], ys)
        for i, (n, r, c) in enumerate(tail):
            qk.gemv(synth.TYPE_IDS[n], Wt[i], r, c, x4.view(1, c), y=yt[i].view(1, r))

    us = _graph_time_us(token, reps=20)
    launches = L * len(groups) + len(tail)
    del Ws, Wt
    torch.cuda.empty_cache()
    return {"workload": "Llama-7B-shaped stack, decode batch 1: 32 layers + lm_head 32000x4096 Q6_K + 2 x 4096^2 Q8_0",
            "weight_bytes": int(nbytes), "us_per_token": round(us, 1),
            "tokens_per_s_equiv": round(1e6 / us, 1), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
            "launches_per_token": launches, "timing": "one CUDA graph per token, median of 20 replays"}


def run_ffn_sweep(dev):
    """Llama-3-8B FFN (gate/up 14336x4096, down 4096x14336) in Q4_K and Q5_0,
    activation batches M in {1, 4, 16, 64}: the fused GEMV (qk_gemv; M = 1
    with gate/up as one qk_gemv_batch) against the tensor-core GEMM (qk_gemm,
    bf16 activations), per M.  Three copies of the weights rotate (beyond
    L2).  GB/s counts packed weights + x + y; TFLOP/s = 2*M*N*K / time."""
    import torch
    import gguf_quant_dequant_gb300 as qk
    import synth
    out = {}
    g = torch.Generator(device=dev)
    g.manual_seed(5252)
    for name in ("Q4_K", "Q5_0"):
        t = synth.TYPE_IDS[name]
        mats = synth.llama3_ffn(name)
        ncop = 3
        Ws = [[synth.random_blocks_torch(name, r, c, 7000 + 10 * k + i, dev) for i, (_, _, r, c) in enumerate(mats)]
              for k in range(ncop)]
        wbytes = sum(w.numel() for w in Ws[0])
        flop1 = sum(2.0 * r * c for (_, _, r, c) in mats)
        res = {}
        for M in synth.FFN_BATCHES:
            X = {c: torch.randn((M, c), device=dev, generator=g) for c in (4096, 14336)}
            Xb = {c: v.to(torch.bfloat16) for c, v in X.items()}
            Y = [torch.empty((M, r), device=dev) for (_, _, r, _) in mats]
            ws = torch.empty(max(16, max(qk.gemv_workspace(t, r, c, M) for (_, _, r, c) in mats)),
                             dtype=torch.uint8, device=dev)

            def gemv_pass():
                for k in range(ncop):
                    if M == 1:
                        qk.gemv_batch(t, Ws[k][0:2], [14336, 14336], 4096, X[4096][0], ys=[Y[0][0], Y[1][0]])
                    else:
                        for i in range(2):
                            qk.gemv(t, Ws[k][i], 14336, 4096, X[4096], y=Y[i], ws=ws)
                    qk.gemv(t, Ws[k][2], 4096, 14336, X[14336], y=Y[2], ws=ws)

            def gemm_pass():
                for k in range(ncop):
                    for i, (_, _, r, c) in enumerate(mats):
                        qk.gemm(t, Ws[k][i], r, c, Xb[c], Y=Y[i])

            us_v = _graph_time_us(gemv_pass) / ncop
            us_m = _graph_time_us(gemm_pass) / ncop
            io = 4 * M * (4096 + 14336) + 4 * M * (2 * 14336 + 4096)
            res[str(M)] = {"gemv_us": round(us_v, 2), "gemm_us": round(us_m, 2),
                           "gemv_gbs": round((wbytes + io) / (us_v * 1e-6) / 1e9, 1),
                           "gemm_gbs": round((wbytes + io) / (us_m * 1e-6) / 1e9, 1),
                           "gemv_tflops": round(M * flop1 / (us_v * 1e-6) / 1e12, 2),
                           "gemm_tflops": round(M * flop1 / (us_m * 1e-6) / 1e12, 2),
                           "faster": "gemv" if us_v <= us_m else "gemm"}
            del X, Xb, Y, ws
        cross = next((int(M) for M, v in res.items() if v["faster"] == "gemm"), None)
        out[name] = {"per_M": res, "weight_bytes": int(wbytes), "gemm_faster_from_M": cross}
        del Ws
        torch.cuda.empty_cache()
    return out


def run_e2e(args, dev, layer, groups, Wd, xs, lb):
    """Same step through the C ABI from pinned HOST buffers: every step copies
    the layer's packed weights and activations host->device, runs the four
    launches and copies the outputs back; all inside the timed region.  The
    copies run on their own stream, one launch group ahead of the compute
    (an event per group), into two sets of device buffers used by alternate
    steps, so the link stays busy while the kernels run.  The host->device
    copy rate of the link is the bound (about 210 GB/s measured)."""
    import torch
    Wh = [w.cpu().pin_memory() for w in Wd]
    xh = [x.cpu().pin_memory() for x in xs]
    yd = [torch.empty(rows, device=dev) for (_, _, rows, _) in layer]
    yh = [torch.empty(rows).pin_memory() for (_, _, rows, _) in layer]
    sets = [([torch.empty_like(w, device=dev) for w in Wd], [torch.empty_like(x, device=dev) for x in xs])
            for _ in range(2)]
    stream = torch.cuda.current_stream()
    copy_s = torch.cuda.Stream()
    done = [torch.cuda.Event(), torch.cuda.Event()]   # compute finished with buffer set k
    for ev in done:
        ev.record(stream)
    state = {"k": 0}

    def step():
        k = state["k"]
        Wdd, xd = sets[k]
        copy_s.wait_event(done[k])            # the step two back has finished reading set k
        ready = []
        with torch.cuda.stream(copy_s):
            for gi, grp in enumerate(groups):
                for i in grp:
                    Wdd[i].copy_(Wh[i], non_blocking=True)
                xd[gi].copy_(xh[gi], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_s)
                ready.append(ev)
        for gi, grp in enumerate(groups):
            stream.wait_event(ready[gi])
            run_group(layer, grp, Wdd, xd[gi], yd)
            for i in grp:
                yh[i].copy_(yd[i], non_blocking=True)
        done[k].record(stream)
        state["k"] = 1 - k

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    n = max(5, min(args.steps, 50))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_s.wait_stream(stream)   # no copy starts before the timed region
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    h2d = sum(w.numel() for w in Wh) + sum(4 * x.numel() for x in xh)
    d2h = sum(4 * y.numel() for y in yh)
    return {"value": round(lb / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": n,
            "transfer": "pinned host buffers, cudaMemcpyAsync on a copy stream one launch group ahead of "
                        "the compute, two device buffer sets alternating by step"}


def _oracle_layer_sample(row_div: int):
    """Host inputs of the layer; with row_div > 1 only the first rows/row_div
    rows of each matrix (a bounded sample of the same workload)."""
    import synth
    mats = []
    for gi, grp in enumerate(synth.LLAMA7B_LAYER_GROUPS):
        cols = synth.LLAMA7B_LAYER[grp[0]][3]
        x = synth.activations(1, cols, 400 + gi)          # one activation vector per launch group
        for k, i in enumerate(grp):
            (nm, name, rows, _) = synth.LLAMA7B_LAYER[i]
            r = max(1, rows // row_div)
            W = synth.random_blocks(name, r, cols, 300 + i)
            mats.append((synth.TYPE_IDS[name], W, r, cols, x,
                         r * synth.row_bytes(name, cols) + 4 * r + (4 * cols if k == 0 else 0)))
    return mats


_BARRIER = None


def _oracle_share_init(barrier):
    global _BARRIER
    _BARRIER = barrier


def _oracle_share(job):
    """One process of the all-core CPU baseline: the oracle as it stands on
    rows k, k + n, ... of every matrix of the layer (its own seeded blocks of
    the same distribution), passes until budget_s; all processes start the
    timed loop together."""
    k, n, budget_s = job
    import oracle
    import synth
    mats = []
    for gi, grp in enumerate(synth.LLAMA7B_LAYER_GROUPS):
        cols = synth.LLAMA7B_LAYER[grp[0]][3]
        x = synth.activations(1, cols, 400 + gi)
        for i in grp:
            (_, name, rows, _) = synth.LLAMA7B_LAYER[i]
            r = rows // n + (1 if k < rows % n else 0)
            if r:
                W = synth.random_blocks(name, r, cols, 3000 + 31 * i + k)
                mats.append((synth.TYPE_IDS[name], W, r, cols, x, r * synth.row_bytes(name, cols)))
    _BARRIER.wait()
    t0 = time.perf_counter()
    nbytes, passes = 0, 0
    while True:
        for (t, W, r, cols, x, b) in mats:
            oracle.gemv(t, W, r, cols, x)
            nbytes += b
        passes += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return nbytes, time.perf_counter() - t0, passes


def cpu_baseline_all_cores(budget_s: float = 10.0):
    """The same oracle on every host core: one spawned process per core, each
    on its share of the layer's rows; GB/s = all bytes / the longest timed
    loop."""
    import multiprocessing as mp
    n = len(os.sched_getaffinity(0))
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(n)
    with ctx.Pool(n, initializer=_oracle_share_init, initargs=(barrier,)) as pool:
        res = pool.map(_oracle_share, [(k, n, budget_s) for k in range(n)])
    nbytes = sum(r[0] for r in res)
    dt = max(r[1] for r in res)
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": n,
            "sample": f"{n} processes, each the layer's 7 GEMVs on 1/{n} of every matrix's rows, "
                      f"{min(r[2] for r in res)}+ passes in {dt:.1f} s"}


def cpu_baseline(layer, budget_s: float = 10.0):
    """The oracle as it stands, single-threaded, on passes over one full layer
    until about budget_s seconds have run; then the same on all host cores."""
    import oracle
    oracle.build()
    mats = _oracle_layer_sample(1)
    t0 = time.perf_counter()
    passes, nbytes = 0, 0
    while True:
        for (t, W, r, cols, x, b) in mats:
            oracle.gemv(t, W, r, cols, x)
            nbytes += b
        passes += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{passes} full pass(es) of the layer's 7 GEMVs (batch 1), scalar C, fp64 accumulation",
            "seconds": round(dt, 2), "all_cores": cpu_baseline_all_cores(budget_s)}


def run_reference(args):
    """The CPU oracle as the reference arm: each step is the layer with every
    matrix cut to its first 1/64 of rows (full K), timed on one host core."""
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    oracle.build()
    mats = _oracle_layer_sample(64)
    sample_bytes = sum(m[5] for m in mats)
    for _ in range(args.warmup):
        for (t, W, r, cols, x, b) in mats:
            oracle.gemv(t, W, r, cols, x)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for (t, W, r, cols, x, b) in mats:
            oracle.gemv(t, W, r, cols, x)
    dt = time.perf_counter() - t0
    ms = dt / args.steps * 1e3
    value = sample_bytes / (ms * 1e-3) / 1e9
    sample = "Llama-7B layer at decode batch 1, first 1/64 of each matrix's rows, scalar C oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "q4_k/q6_k blocks, f64 accumulation",
        "data": "synthetic (seeded random blocks, x ~ N(0,1))",
        "config": {"workload": "Llama-7B-shaped decoder layer, decode batch 1: q/k/v/o 4096x4096 Q4_K, "
                               "gate/up 11008x4096 Q4_K, down 4096x11008 Q6_K",
                   "bytes_per_step": sample_bytes, "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="qk", choices=["qk", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--no-gemm", action="store_true", help="skip the prefill GEMM leg")
    ap.add_argument("--no-stack", action="store_true", help="skip the 32-layer stack leg")
    ap.add_argument("--no-sweep", action="store_true", help="skip the Llama-3 FFN batch sweep")
    ap.add_argument("--gemm-only", action="store_true",
                    help="run only the prefill GEMM leg and print its JSON (for profiling)")
    ap.add_argument("--no-quant", action="store_true", help="skip the quantizer leg")
    ap.add_argument("--record-traffic", metavar="CSV",
                    help="write the decode kernel's DRAM-traffic record from the launch list of its ncu command")
    ap.add_argument("--no-swiglu", action="store_true", help="skip the fused SwiGLU leg")
    ap.add_argument("--no-attn", action="store_true", help="skip the quantized-KV attention leg")
    ap.add_argument("--no-codes-check", action="store_true",
                    help="skip timing the layer a second time on random-byte codes")
    ap.add_argument("--attn-only", action="store_true", help="run the quantized-KV attention leg alone")
    ap.add_argument("--swiglu-only", action="store_true",
                    help="run only the fused SwiGLU leg and print its JSON (for profiling)")
    ap.add_argument("--quantize-only", action="store_true",
                    help="run only the quantizer leg and print its JSON (for profiling)")
    ap.add_argument("--ffn-gemm", type=int, default=0, metavar="M",
                    help="run only the small-batch GEMM over the Llama-3 FFN at batch M (for profiling)")
    ap.add_argument("--min-warmup-s", type=float, default=1.0,
                    help="keep replaying warm-up steps for at least this long (clocks settle)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.record_traffic:
        print(json.dumps(record_traffic(args.record_traffic)))
        return
    if args.impl == "reference":
        run_reference(args)
    elif args.gemm_only or args.ffn_gemm > 0 or args.quantize_only or args.swiglu_only or args.attn_only:
        import torch
        from gguf_quant_dequant_gb300 import build as qkbuild
        qkbuild.build()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        if args.swiglu_only:
            print(json.dumps(run_swiglu(dev)))
        elif args.attn_only:
            print(json.dumps(run_attn(dev)))
        elif args.quantize_only:
            print(json.dumps(run_quantize(dev, reps=args.steps)))
        elif args.ffn_gemm > 0:
            print(json.dumps(run_ffn_gemm(dev, args.ffn_gemm, reps=args.steps)))
        else:
            print(json.dumps(run_gemm_bench(dev, reps=args.steps)))
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
