"""Benchmark of the Q1 (1-bit affine, group size 128) linear layer on GB300.

Headline workload (decode QMV, M = 1, 27B-class shapes): one decode step is one
token through a stack of 64 layers, each with four Q1 projections
  gate  [17408 x 5120]   up [17408 x 5120]   down [5120 x 17408]   attn [5120 x 5120]
with symmetric metadata (bias derived, not stored) and bf16 activations ~N(0,1).
The 64 layers hold 2.64 GB of packed weights and scales, 20x the 129 MB L2, so
every step streams its weights from HBM (no flush needed).  A step is replayed
as a CUDA graph of the library's public calls.

  value      achieved HBM GB/s = algorithmic bytes of the step / device time
             (packed words + fp16 metadata + x + y, each once)
  e2e        the same metric with the step's activations copied in from pinned
             host memory and its outputs copied back inside the timed region
  roofline   the narrow kernel (the only kernel of the step) against the
             measured HBM copy bandwidth
  sub        narrow M = 2..8 GB/s, the affine variant, and prefill TFLOP/s

`--impl reference` times the CPU oracle (the only reference implementation:
the pages publish no code) on the same metric and a bounded sample.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

LAYERS = 64
D_MODEL, D_FF = 5120, 17408
VOCAB = 152064  # 27B-class vocabulary: embedding table and tied head [VOCAB x D_MODEL]
SHAPES = (("gate", D_FF, D_MODEL), ("up", D_FF, D_MODEL), ("down", D_MODEL, D_FF),
          ("attn", D_MODEL, D_MODEL))
WORKLOAD = "q1 decode QMV M=1, 64 layers x {gate,up 17408x5120; down 5120x17408; attn 5120x5120}, symmetric g128"

# DRAM traffic per launch of the narrow kernel on the gate shape (17408 x 5120,
# M = 1), from ncu (dram__bytes_read.sum + dram__bytes_write.sum), and the
# sha256 of q1_narrow.cu it was taken on; reported as null once the source differs.
NCU_TRAFFIC = {"bytes": 12595968, "source_sha256": "0201254629d1d1b5ea93a42192705cbc0d0d9ed479514163062b1f3d6e07356e"}


def weight_bytes(N, K, affine):
    G = K // 128
    return N * K // 8 + N * G * 2 * (2 if affine else 1)


def step_bytes(M, affine=False):
    tot = 0
    for _, N, K in SHAPES:
        tot += weight_bytes(N, K, affine) + M * K * 2 + M * N * 2
    return tot * LAYERS


def chain_bytes(M):
    """Algorithmic bytes of one token of the decode chain: every weight once;
    per layer h and a in/out of the attention product, a in and the FFN
    intermediate out of the gate/up launch, the intermediate in and h out of
    the down launch (bf16)."""
    w = sum(weight_bytes(N, K, False) for _, N, K in SHAPES)
    act = M * 2 * (4 * D_MODEL + 2 * D_FF)
    return (w + act) * LAYERS


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "utilization.gpu")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        """Median SM clock over the samples taken under load (GPU utilization
        >= 50 %; all samples if none is), the maximum clock, every throttle
        reason seen active, and both sample counts."""
        sm, mx, busy, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [c.strip() for c in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                clk, cmax = float(p[0]), float(p[1])
            except ValueError:
                continue
            sm.append(clk)
            mx.append(cmax)
            try:
                if float(p[8]) >= 50.0:
                    busy.append(clk)
            except ValueError:
                pass
            for nm, v in zip(names, p[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_under_load": 0}
        return {"sm_mhz": statistics.median(busy or sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm), "samples_under_load": len(busy),
                "sample_period_ms": 100}


# ---------------------------------------------------------------------------
# CPU oracle timing (runs in a child process pinned to one thread)
# ---------------------------------------------------------------------------
def cpu_worker(seconds: float):
    import numpy as np
    from bit_affine_quantized_g128_gb300 import synth
    from oracle import q1_oracle as O
    N, K = D_FF, D_MODEL
    rows_per_chunk = 256
    t = synth.q1_tensor(2048, K, seed=1001, affine=False)
    x = synth.activations(1, K, seed=1006)
    done_bytes, done_rows = 0, 0
    t0 = time.perf_counter()
    i = 0
    while time.perf_counter() - t0 < seconds:
        r0 = (i * rows_per_chunk) % 2048
        sl = slice(r0, r0 + rows_per_chunk)
        O.qmm(x, t.words[sl], t.scales[sl], None, K)
        done_rows += rows_per_chunk
        done_bytes += weight_bytes(rows_per_chunk, K, False) + K * 2 + rows_per_chunk * 2
        i += 1
    el = time.perf_counter() - t0
    print(json.dumps({"bytes": done_bytes, "seconds": el, "rows": done_rows}))


def cpu_baseline(seconds: float):
    # the oracle on every host core: its BLAS thread count is fixed to the
    # core count before numpy loads in the child, and the line reports it
    cores = os.cpu_count() or 1
    env = dict(os.environ, OMP_NUM_THREADS=str(cores), OPENBLAS_NUM_THREADS=str(cores),
               MKL_NUM_THREADS=str(cores), CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", str(seconds)],
                       capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return {"value": None, "unit": "GB/s", "cores": cores, "kind": "oracle",
                "sample": f"failed: {r.stderr.strip()[-200:]}"}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": d["bytes"] / d["seconds"] / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": (f"oracle QMV M=1 on {d['rows']} rows of a symmetric 17408x5120 gate matrix "
                       f"(chunks of 256 rows, {d['seconds']:.1f} s, BLAS on {cores} threads); GB/s of "
                       "the same algorithmic bytes per row as the GPU metric")}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def build_stack(q1, synth, torch, device, affine, seed0, meta_bf16=False):
    layers = []
    for li in range(LAYERS):
        ws = {}
        for j, (name, N, K) in enumerate(SHAPES):
            sd = seed0 + 4 * li + j
            w = synth.device_weight_words(N, K, sd, device)
            s = synth.device_scales(N, K, sd + 7919, device)
            b = synth.device_biases(N, K, sd + 15485863, device) if affine else None
            if meta_bf16:  # the same draws rounded to bf16
                s = s.to(torch.bfloat16)
                b = None if b is None else b.to(torch.bfloat16)
            ws[name] = q1.Q1Weight(w, s, b, K)
        layers.append(ws)
    return layers


def make_step(q1, torch, layers, M, device):
    xs, ys = [], []
    g = torch.Generator(device=device)
    g.manual_seed(1006 + M)
    for ws in layers:
        for name, N, K in SHAPES:
            xs.append(torch.randn((M, K), generator=g, device=device).to(torch.bfloat16))
            ys.append(torch.empty((M, N), dtype=torch.bfloat16, device=device))

    def step():
        i = 0
        for ws in layers:
            for name, N, K in SHAPES:
                if M == 1:
                    q1.qmv(ws[name], xs[i], out=ys[i].view(N))
                else:
                    q1.qmm_narrow(ws[name], xs[i], out=ys[i])
                i += 1
    return step, xs, ys


def time_graph(torch, step, warmup, steps, stream):
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    return graph


def run_timed(torch, graph, steps, stream, dist=None):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return e0.elapsed_time(e1) / 1e3  # seconds


def graph_time(torch, fns, stream, per=10, reps=5):
    """Seconds per call: `per` calls (cycling over `fns`) captured in one CUDA
    graph, replayed `reps` times after 3 warm-up replays."""
    gm = time_graph(torch, lambda: [fns[i % len(fns)]() for i in range(per)], 3, 3, stream)
    t = run_timed(torch, gm, reps, stream) / (reps * per)
    del gm
    return t


def elementwise_and_head(q1, synth, torch, device, stream):
    """GB/s of algorithmic bytes for the tied head (QMV over the vocabulary),
    dequantize, pack, unpack and the symmetric check, and the time of a 64-id
    embedding gather.  Inputs rotate over more than the 129 MB L2 where the
    work is a stream."""
    out = {}
    G = D_MODEL // 128
    # tied head: two vocabulary matrices in turn (2 x 109.5 MB)
    heads = [q1.Q1Weight(synth.device_weight_words(VOCAB, D_MODEL, 4400 + i, device),
                         synth.device_scales(VOCAB, D_MODEL, 4410 + i, device), None, D_MODEL) for i in range(2)]
    xh = torch.randn(D_MODEL, device=device).to(torch.bfloat16)
    yh = torch.empty(VOCAB, dtype=torch.bfloat16, device=device)
    t = graph_time(torch, [lambda W=W: q1.qmv(W, xh, out=yh) for W in heads], stream)
    out["tied_head_152064x5120_GBps"] = round((weight_bytes(VOCAB, D_MODEL, False) + D_MODEL * 2 + VOCAB * 2) / t / 1e9, 1)
    # embedding gather: 64 ids into the table (latency-bound: 46 KB read, 655 KB written)
    ids = torch.randint(0, VOCAB, (64,), device=device, dtype=torch.int32)
    t = graph_time(torch, [lambda: q1.embed_gather(heads[0], ids)], stream)
    out["embed_gather_T64_us"] = round(t * 1e6, 2)
    out["embed_gather_T64_GBps"] = round(64 * (D_MODEL // 8 + G * 2 + D_MODEL * 2) / t / 1e9, 1)
    # dequantize a 17408 x 5120 projection to bf16 (178 MB written)
    W1 = q1.Q1Weight(synth.device_weight_words(D_FF, D_MODEL, 4420, device),
                     synth.device_scales(D_FF, D_MODEL, 4421, device), None, D_MODEL)
    t = graph_time(torch, [lambda: q1.dequantize(W1, torch.bfloat16)], stream)
    out["dequantize_bf16_17408x5120_GBps"] = round((weight_bytes(D_FF, D_MODEL, False) + D_FF * D_MODEL * 2) / t / 1e9, 1)
    # unpack / pack of two stacked projections (2 x 17408 rows: 178 MB of bits)
    words = torch.cat([W1.words, heads[1].words[:D_FF]])
    bits = q1.unpack(words, D_MODEL)
    nbytes = words.numel() * 4 + bits.numel()
    t = graph_time(torch, [lambda: q1.unpack(words, D_MODEL)], stream)
    out["unpack_34816x5120_GBps"] = round(nbytes / t / 1e9, 1)
    t = graph_time(torch, [lambda: q1.pack(bits)], stream)
    out["pack_34816x5120_GBps"] = round(nbytes / t / 1e9, 1)
    del bits, words, W1
    # symmetric check of stored biases: six vocabulary-sized metadata sets in
    # turn (6 x 24 MB of scales and biases)
    metas = []
    for i in range(6):
        # scales >= 2^-13 so that -scale/2 is a normal fp16 value (exact)
        sc = synth.device_scales(VOCAB, D_MODEL, 4430 + i, device).clamp(min=2.0 ** -13)
        metas.append(q1.Q1Weight(heads[0].words, sc, (sc.float() * -0.5).to(torch.float16), D_MODEL))
    t = graph_time(torch, [lambda W=W: q1.check_symmetric(W) for W in metas], stream, per=12)
    out["check_symmetric_152064x5120_GBps"] = round(VOCAB * G * 4 / t / 1e9, 1)
    assert all(int(q1.check_symmetric(W).item()) == 1 for W in metas)
    del metas, heads
    return out


def time_prefill(q1, synth, torch, device, M, shape, affine, reps=20):
    name, N, K = shape
    nl = 6  # rotate over weights + activations larger than L2
    Ws = [q1.Q1Weight(synth.device_weight_words(N, K, 77 + i, device),
                      synth.device_scales(N, K, 177 + i, device),
                      synth.device_biases(N, K, 277 + i, device) if affine else None, K)
          for i in range(nl)]
    g = torch.Generator(device=device)
    g.manual_seed(1004)
    xs = [torch.randn((M, K), generator=g, device=device).to(torch.bfloat16) for _ in range(nl)]
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device=device) for _ in range(nl)]
    ws = q1.qmm_workspace(M, N, K, device)
    for i in range(nl):
        q1.qmm(Ws[i], xs[i], workspace=ws, out=ys[i])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for r in range(reps):
        i = r % nl
        q1.qmm(Ws[i], xs[i], workspace=ws, out=ys[i])
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / reps
    # unfused comparator: dequantize to bf16, then a dense bf16 GEMM (cuBLAS via
    # torch), over the same rotation of weights and activations (larger than L2)
    for i in range(nl):
        torch.matmul(xs[i], q1.dequantize(Ws[i], torch.bfloat16).T, out=ys[i])
    torch.cuda.synchronize()
    e0.record()
    for r in range(reps):
        i = r % nl
        tmp = q1.dequantize(Ws[i], torch.bfloat16)
        torch.matmul(xs[i], tmp.T, out=ys[i])
    e1.record()
    torch.cuda.synchronize()
    t_unfused = e0.elapsed_time(e1) / 1e3 / reps
    del Ws, xs, ys
    return 2.0 * M * N * K / t / 1e12, 2.0 * M * N * K / t_unfused / 1e12


def weight_bytes_g(N, K, affine, group):
    """Algorithmic bytes of one packed matrix with metadata per `group` weights."""
    G = K // group
    return N * K // 8 + N * G * 2 * (2 if affine else 1)


def narrow_sweep(q1, synth, torch, device, stream):
    """GB/s of single launches (graph of launches over 12 distinct matrices,
    150-210 MB, more than the L2) on the two 27B-class FFN shapes: M = 1..9,
    12, 16 and 17 (9..16 run as two narrow launches at the default
    threshold, 17 on the prefill path), symmetric and affine; and M = 1 with
    metadata per 64 and per 32 weights."""
    out = {}
    nl = 12
    for name, N, K in (SHAPES[0], SHAPES[2]):
        for affine in (False, True):
            Ws = [q1.Q1Weight(synth.device_weight_words(N, K, 300 + i, device),
                              synth.device_scales(N, K, 320 + i, device),
                              synth.device_biases(N, K, 340 + i, device) if affine else None, K)
                  for i in range(nl)]
            ws = q1.qmm_workspace(17, N, K, device)
            for M in list(range(1, 10)) + [12, 16, 17]:
                x = torch.randn((M, K), device=device).to(torch.bfloat16)
                y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
                t = graph_time(torch, [lambda W=W: q1.qmm(W, x, workspace=ws, out=y) for W in Ws], stream, per=24)
                b = weight_bytes(N, K, affine) + M * K * 2 + M * N * 2
                out[f"qmm_{name}_{'affine' if affine else 'sym'}_M{M}_GBps"] = round(b / t / 1e9, 1)
            del Ws
            torch.cuda.empty_cache()
    name, N, K = SHAPES[0]
    for group in (64, 32):
        Ws = []
        for i in range(nl):
            g = torch.Generator(device=device)
            g.manual_seed(360 + i)
            sc = (torch.randn((N, K // group), generator=g, device=device).abs() * 0.02 + 1e-4).to(torch.float16)
            Ws.append(q1.Q1Weight(synth.device_weight_words(N, K, 350 + i, device), sc, None, K))
        x = torch.randn((K,), device=device).to(torch.bfloat16)
        y = torch.empty((N,), dtype=torch.bfloat16, device=device)
        t = graph_time(torch, [lambda W=W: q1.qmv(W, x, out=y) for W in Ws], stream, per=24)
        out[f"qmv_{name}_group{group}_M1_GBps"] = round((weight_bytes_g(N, K, False, group) + K * 2 + N * 2) / t / 1e9, 1)
        del Ws
        torch.cuda.empty_cache()
    return out


def ffn_bytes(M, affine=False):
    """Algorithmic bytes of one fused FFN call: the three matrices once, x in,
    the bf16 intermediate h written and read, y out."""
    w = 2 * weight_bytes(D_FF, D_MODEL, affine) + weight_bytes(D_MODEL, D_FF, affine)
    return w + M * D_MODEL * 2 + 2 * M * D_FF * 2 + M * D_MODEL * 2


def ffn_sweep(q1, synth, torch, device, stream):
    """GB/s of q1_ffn_fused at M = 1, 4, 8 over 6 distinct FFN blocks (226 MB)."""
    out = {}
    blocks = []
    for i in range(6):
        mk = lambda N, K, sd: q1.Q1Weight(synth.device_weight_words(N, K, sd, device),
                                          synth.device_scales(N, K, sd + 1, device), None, K)
        blocks.append((mk(D_FF, D_MODEL, 400 + 10 * i), mk(D_FF, D_MODEL, 402 + 10 * i), mk(D_MODEL, D_FF, 404 + 10 * i)))
    for M in (1, 4, 8):
        x = torch.randn((M, D_MODEL), device=device).to(torch.bfloat16)
        y = torch.empty((M, D_MODEL), dtype=torch.bfloat16, device=device)
        ws = q1.ffn_workspace(M, D_MODEL, D_FF, device)
        t = graph_time(torch, [lambda B=B: q1.ffn_fused(*B, x, workspace=ws, out=y) for B in blocks], stream, per=12)
        out[f"ffn_fused_M{M}_GBps"] = round(ffn_bytes(M) / t / 1e9, 1)
        out[f"ffn_fused_M{M}_us"] = round(t * 1e6, 2)
    del blocks
    torch.cuda.empty_cache()
    return out


def profile_case(args):
    """A few launches of one kernel on one shape, for ncu (small device footprint)."""
    import torch
    from bit_affine_quantized_g128_gb300 import build as qbuild
    from bit_affine_quantized_g128_gb300 import q1, synth
    qbuild.build()
    q1.load_library()
    device = torch.device("cuda", 0)
    case = args.profile
    if case.startswith("decode") or case.startswith("narrow"):
        M = 1 if case.startswith("decode") else int(case.split("M")[-1])
        shape = {"gate": SHAPES[0], "down": SHAPES[2], "attn": SHAPES[3]}[args.shape]
        _, N, K = shape
        nl = 12  # > L2 in total: 12 x 12.5 MB
        Ws = [q1.Q1Weight(synth.device_weight_words(N, K, 11 + i, device),
                          synth.device_scales(N, K, 111 + i, device), None, K) for i in range(nl)]
        x = torch.randn((M, K), device=device).to(torch.bfloat16)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        for r in range(args.steps):
            q1.qmm_narrow(Ws[r % nl], x, out=y)
    elif case.startswith("ffn"):  # fused FFN: narrow_kernel<2> gate/up, then the down projection
        M = int(case.split("M")[-1])
        nl = 4  # 4 x 62.9 MB of FFN weights: more than the L2
        ffns = [[q1.Q1Weight(synth.device_weight_words(N, K, 21 + 3 * i + j, device),
                             synth.device_scales(N, K, 121 + 3 * i + j, device), None, K)
                 for j, (_, N, K) in enumerate((SHAPES[0], SHAPES[1], SHAPES[2]))] for i in range(nl)]
        x = torch.randn((M, D_MODEL), device=device).to(torch.bfloat16)
        y = torch.empty((M, D_MODEL), dtype=torch.bfloat16, device=device)
        ws = q1.ffn_workspace(M, D_MODEL, D_FF, device)
        for r in range(args.steps):
            g, u, d = ffns[r % nl]
            q1.ffn_fused(g, u, d, x, workspace=ws, out=y)
    elif case == "elementwise":  # dequantize, unpack, pack, gather, symmetric check, repack, once each
        W1 = q1.Q1Weight(synth.device_weight_words(D_FF, D_MODEL, 31, device),
                         synth.device_scales(D_FF, D_MODEL, 131, device), None, D_MODEL)
        sc = synth.device_scales(D_FF, D_MODEL, 231, device).clamp(min=2.0 ** -13)
        Wb = q1.Q1Weight(W1.words, sc, (sc.float() * -0.5).to(torch.float16), D_MODEL)
        ids = torch.randint(0, D_FF, (64,), device=device, dtype=torch.int32)
        for r in range(args.steps):
            dense = q1.dequantize(W1, torch.bfloat16)
            bits = q1.unpack(W1.words, D_MODEL)
            q1.pack(bits)
            q1.embed_gather(W1, ids)
            q1.check_symmetric(Wb)
            q1.pack_from_dense(dense, symmetric=True)
            del dense, bits
    else:  # prefill
        M = int(case.split("M")[-1])
        _, N, K = {"gate": SHAPES[0], "down": SHAPES[2], "attn": SHAPES[3]}[args.shape]
        W = q1.Q1Weight(synth.device_weight_words(N, K, 11, device), synth.device_scales(N, K, 111, device), None, K)
        x = torch.randn((M, K), device=device).to(torch.bfloat16)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        ws = q1.qmm_workspace(M, N, K, device)
        for r in range(args.steps):
            q1.qmm(W, x, workspace=ws, out=y)
    torch.cuda.synchronize()
    assert q1.device_errors() == 0
    print("profile case done", case, args.shape)


def gpu_arm(args):
    import torch
    from bit_affine_quantized_g128_gb300 import build as qbuild
    from bit_affine_quantized_g128_gb300 import q1, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if rank == 0:
        qbuild.build()
    if dist is not None:
        dist.barrier()
    q1.load_library()

    stream = torch.cuda.Stream(device=device)
    layers = build_stack(q1, synth, torch, device, affine=False, seed0=5000 + 1000 * rank)
    torch.cuda.synchronize()

    # ---- headline: decode M = 1
    step, xs, ys = make_step(q1, torch, layers, 1, device)
    graph = time_graph(torch, step, args.warmup, args.steps, stream)
    with ClockSampler(local) as clk:
        secs = run_timed(torch, graph, args.steps, stream, dist)
    clocks = clk.summary()
    bytes_step = step_bytes(1)
    value, t_max, _ = aggregate_over_ranks(bytes_step * args.steps, secs, dist, device)
    launches = args.steps * LAYERS * len(SHAPES)

    # ---- e2e: inputs from pinned host memory, outputs back, every step
    x_host = torch.empty(sum(x.numel() for x in xs), dtype=torch.bfloat16).pin_memory()
    y_host = torch.empty(sum(y.numel() for y in ys), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x_host, device=device)
    y_dev = torch.empty_like(y_host, device=device)
    # the graph's x/y buffers are views into one flat device buffer each
    off = 0
    for x in xs:
        n = x.numel()
        x_dev[off:off + n].copy_(x.reshape(-1))
        off += n
    x_host.copy_(x_dev.cpu())
    x_views, y_views, off, offy = [], [], 0, 0
    for x, y in zip(xs, ys):
        x_views.append(x_dev[off:off + x.numel()].view(x.shape))
        y_views.append(y_dev[offy:offy + y.numel()].view(y.shape))
        off += x.numel()
        offy += y.numel()

    def step_e2e():
        i = 0
        for ws in layers:
            for name, N, K in SHAPES:
                q1.qmv(ws[name], x_views[i], out=y_views[i].view(N))
                i += 1
    g2 = time_graph(torch, step_e2e, 2, 2, stream)
    e2e_steps = max(10, args.steps // 10)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            x_dev.copy_(x_host, non_blocking=True)
            g2.replay()
            y_host.copy_(y_dev, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = e0.elapsed_time(e1) / 1e3
    e2e_value, _, _ = aggregate_over_ranks(bytes_step * e2e_steps, t_e2e, dist, device)
    e2e = {"value": round(e2e_value, 1), "unit": "GB/s",
           "h2d_bytes_per_step": x_host.numel() * 2, "d2h_bytes_per_step": y_host.numel() * 2,
           "path": "q1_qmv calls captured in a CUDA graph; x copied from pinned host and y back every step"}
    del g2, graph

    sub = {}
    if not args.quick:
        # narrow M = 2..8 (same stack), GB/s
        for M in (2, 4, 8):
            stp, _, _ = make_step(q1, torch, layers, M, device)
            gm = time_graph(torch, stp, 3, 3, stream)
            n = max(20, args.steps // 10)
            s_ = run_timed(torch, gm, n, stream)
            sub[f"narrow_M{M}_GBps"] = round(step_bytes(M) * n / s_ / 1e9, 1)
            del gm
        # the synthetic decode chain over the same 64 layers (attention-like
        # product, then the fused FFN; 192 dependent launches per token), M = 1
        chain = [(ws["attn"], ws["gate"], ws["up"], ws["down"]) for ws in layers]
        gc = torch.Generator(device=device)
        gc.manual_seed(1010)
        xc = torch.randn((1, D_MODEL), generator=gc, device=device).to(torch.bfloat16)
        yc = torch.empty_like(xc)
        wsc = q1.decode_chain_workspace(1, D_MODEL, D_FF, device)
        gm = time_graph(torch, lambda: q1.decode_chain(chain, xc, workspace=wsc, out=yc), 3, 3, stream)
        n = max(20, args.steps // 10)
        s_ = run_timed(torch, gm, n, stream)
        sub["decode_chain_ms_per_token"] = round(s_ / n * 1e3, 4)
        sub["decode_chain_GBps"] = round(chain_bytes(1) * n / s_ / 1e9, 1)
        del gm, chain
        del layers
        torch.cuda.empty_cache()
        # affine metadata (bias stored): M = 1
        la = build_stack(q1, synth, torch, device, affine=True, seed0=9000)
        stp, _, _ = make_step(q1, torch, la, 1, device)
        gm = time_graph(torch, stp, 3, 3, stream)
        n = max(20, args.steps // 10)
        s_ = run_timed(torch, gm, n, stream)
        sub["affine_M1_GBps"] = round(step_bytes(1, True) * n / s_ / 1e9, 1)
        del gm, la
        torch.cuda.empty_cache()
        # bf16 scales (the Bonsai image checkpoint's metadata type), M = 1
        lb = build_stack(q1, synth, torch, device, affine=False, seed0=9500, meta_bf16=True)
        stp, _, _ = make_step(q1, torch, lb, 1, device)
        gm = time_graph(torch, stp, 3, 3, stream)
        s_ = run_timed(torch, gm, n, stream)
        sub["bf16_meta_M1_GBps"] = round(step_bytes(1) * n / s_ / 1e9, 1)
        del gm, lb
        torch.cuda.empty_cache()
        # exact repack of a dense bf16 projection (17408 x 5120) into Q1:
        # GB/s of the dense read plus the words and scales written
        W0 = q1.Q1Weight(synth.device_weight_words(D_FF, D_MODEL, 4242, device),
                         synth.device_scales(D_FF, D_MODEL, 4243, device), None, D_MODEL)
        dense = q1.dequantize(W0, torch.bfloat16)
        bad = torch.zeros((1,), dtype=torch.int32, device=device)
        Wr = q1.Q1Weight(torch.empty_like(W0.words), torch.empty_like(W0.scales), None, D_MODEL)
        per = 10  # calls per graph replay
        gm = time_graph(torch, lambda: [q1.pack_from_dense(dense, True, bad=bad, out=Wr) for _ in range(per)],
                        3, 3, stream)
        reps = 5
        t_rp = run_timed(torch, gm, reps, stream) / (reps * per)
        assert int(bad.item()) == 0 and torch.equal(Wr.words, W0.words)
        del gm
        rp_bytes = D_FF * D_MODEL * 2 + weight_bytes(D_FF, D_MODEL, False)
        sub["repack_bf16_17408x5120_GBps"] = round(rp_bytes / t_rp / 1e9, 1)
        del W0, dense, Wr
        torch.cuda.empty_cache()
        sub.update(elementwise_and_head(q1, synth, torch, device, stream))
        torch.cuda.empty_cache()
        # narrow M = 1..9 (and the crossover), group sizes 64/32, standalone FFN
        sub.update(narrow_sweep(q1, synth, torch, device, stream))
        sub.update(ffn_sweep(q1, synth, torch, device, stream))
        # prefill on the tensor cores, symmetric and affine, against the
        # unfused dequantize + cuBLAS comparator
        for M in (128, 512, 2048):
            for shp in (SHAPES[0], SHAPES[2]):
                for affine in (False, True):
                    tf, tf_unf = time_prefill(q1, synth, torch, device, M, shp, affine=affine)
                    tag = f"prefill_M{M}_{shp[0]}" + ("_affine" if affine else "")
                    sub[f"{tag}_TFLOPs"] = round(tf, 1)
                    sub[f"{tag}_unfused_TFLOPs"] = round(tf_unf, 1)
                    torch.cuda.empty_cache()
    assert q1.device_errors() == 0, "device-side wait ran out"

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except Exception:
        pass
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    if not peak:
        peak = 6800.0
    src = os.path.join(ROOT, "bit_affine_quantized_g128_gb300", "csrc", "q1_narrow.cu")
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    traffic = NCU_TRAFFIC["bytes"] if NCU_TRAFFIC["source_sha256"] == sha else None
    per_launch_bytes = bytes_step / (LAYERS * len(SHAPES))
    per_launch_s = secs / (args.steps * LAYERS * len(SHAPES))
    achieved = per_launch_bytes / per_launch_s / 1e9
    line = {
        "metric": "Q1 QMV achieved HBM GB/s (% of 8 TB/s) at M=1..8; prefill QMM TFLOP/s",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_max / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded uniform bits, |N(0,0.02)|+1e-4 fp16 scales, N(0,1) bf16 x)",
        "config": {"workload": WORKLOAD, "layers": LAYERS, "M": 1, "metadata": "symmetric",
                   "bytes_per_step": bytes_step,
                   "l2": "inputs larger than L2 (2.64 GB of weights per step, no flush)",
                   "parallelism": f"replicas x{world}"},
        "pct_of_8TBps": round(100 * value / world / 8000.0, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 3), "traffic": traffic,
                     "peak_source": peak_src,
                     "kernel": "narrow_kernel<1,false,true,0> (mma.sync bf16, 8 K-warps of 4-5 groups, producer warp)",
                     "achieved_from": "graph time / launches (launch gaps included)"},
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": launches,
        "sub": sub,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def aggregate_over_ranks(bytes_per_rank: float, secs: float, dist=None, device=None):
    """Whole-job GB/s across ranks: total bytes of all ranks / the slowest
    rank's time (the max over ranks), as every rank processes its own replica."""
    world, t_max, tot = 1, secs, bytes_per_rank
    if dist is not None and dist.is_initialized():
        import torch
        world = dist.get_world_size()
        tt = torch.tensor([secs, bytes_per_rank], dtype=torch.float64, device=device)
        t = tt[:1].clone()
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        b = tt[1:].clone()
        dist.all_reduce(b, op=dist.ReduceOp.SUM)
        t_max, tot = float(t.item()), float(b.item())
    return tot / t_max / 1e9, t_max, world


def reference_arm(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    from bit_affine_quantized_g128_gb300 import synth
    from oracle import q1_oracle as O
    # each step: a bounded sample of the decode workload (256 rows of the gate
    # matrix, M = 1), timed on the host cores; GB/s of the same algorithmic bytes
    K = D_MODEL
    t = synth.q1_tensor(256, K, seed=1001, affine=False)
    x = synth.activations(1, K, seed=1006)
    for _ in range(args.warmup):
        O.qmm(x, t.words, t.scales, None, K)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.qmm(x, t.words, t.scales, None, K)
    el = time.perf_counter() - t0
    b = (weight_bytes(256, K, False) + K * 2 + 256 * 2) * args.steps
    v = b / el / 1e9
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    line = {"metric": "Q1 QMV achieved HBM GB/s (% of 8 TB/s) at M=1..8; prefill QMM TFLOP/s",
            "value": round(v, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "M": 1, "metadata": "symmetric"},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": "each step: oracle QMV on 256 rows of a 17408x5120 symmetric matrix"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline only (no sub-measurements)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-worker", type=float, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--profile", default=None,
                    help="run a few launches of one case for ncu: decode | narrowM<m> | prefillM<m> | ffnM<m> | elementwise")
    ap.add_argument("--shape", default="gate", choices=["gate", "down", "attn"])
    args = ap.parse_args()
    if args.cpu_worker is not None:
        cpu_worker(args.cpu_worker)
        return
    if args.profile:
        profile_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        # numpy is not imported yet: fix the BLAS thread count to the host's
        # cores, so that the line's `cores` is the count the oracle ran with
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = str(os.cpu_count() or 1)
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
