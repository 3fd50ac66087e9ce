"""Benchmark: speculative-decoding verify rounds on Qwen-shaped quantized targets.

A step is one whole verify round: every layer's q|k|v, o, gate|up and down
projections (group-64 affine codes) with the RMSNorm / residual / SwiGLU steps
fused, the 151936-row vocab head with its row statistics, and the accept step
(drafts and draft probabilities given).  Each round is captured once into a
CUDA graph and replayed; the weights are far larger than L2, so no flush is
needed between rounds.

Headline (the JSON line's value): microseconds per round of the Qwen3-8B-shaped
8-bit target at M = 8 rows (anchor + 7 drafts), T = 0.7; the same line carries
M = 1 and 16, the weight-stream bandwidth against the measured HBM copy rate
and 8 TB/s, the cost ratio t(M)/t(1), the spread of single replays, and (unless
--quick) these workloads:

  * sweep_4b: the Qwen3-4B-shaped 4-bit round at every M = 1..32 (the cost
    knee and the draft cap the cap controller picks from that curve), next to
    the same shapes with bf16 weights through cuBLAS;
  * batched_27b: a 27B-class 8-bit round, 64 layers, B = 4 requests x 8 rows,
    T = 1.0, per-request Philox streams;
  * projections: single projections (one-layer 8B shapes at M = 1..17, the
    tiny 4-bit layer at M = 1..8), rotating >= 2 x L2 of weight copies;
  * wide: the tensor-memory (tcgen05) matmul at M = 512 on 8B shapes.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--quick]
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per verify round and weight-stream HBM GB/s (% of peak) at M=1/8/16"
SHAPE_8B = dict(hidden=4096, q_dim=4096, kv_dim=1024, inter=12288, vocab=151936, n_layers=36, bits=8)
SHAPE_4B = dict(hidden=2560, q_dim=4096, kv_dim=1024, inter=9728, vocab=151936, n_layers=36, bits=4)
SHAPE_27B = dict(hidden=5120, q_dim=6144, kv_dim=1024, inter=17408, vocab=151936, n_layers=64, bits=8)
TEMPERATURE = 0.7
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 2 ** 20


def weight_bytes(shape):
    h, dq, kv, i, v, L, bits = (shape[k] for k in ("hidden", "q_dim", "kv_dim", "inter", "vocab", "n_layers", "bits"))
    per_weight = bits / 8 + 4 / 64
    layer = (dq + 2 * kv) * h + h * dq + 2 * i * h + h * i
    return (L * layer + v * h) * per_weight


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


def spread(us):
    s = sorted(us)
    pick = lambda f: s[min(len(s) - 1, int(round(f * (len(s) - 1))))]
    return {"median": round(statistics.median(s), 2), "p10": round(pick(0.1), 2), "p90": round(pick(0.9), 2),
            "mean": round(statistics.fmean(s), 2), "n": len(s)}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.path = index, None, None

    def __enter__(self):
        import tempfile
        self.path = tempfile.mktemp(suffix=".csv")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            self.proc.wait()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 7 and parts[0].replace(".", "").isdigit():
                    rows.append(parts)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][1]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())}


# --------------------------------------------------------------- our path
class Round:
    """Device model, buffers and the captured graph of one verify round.

    rows_per_request: the M rows of one request (anchor + drafts); B requests
    stack their rows; request b's uniforms are Philox stream (seed, b)."""

    def __init__(self, lib, layers, head, shape, rows_per_request, B, seed, temperature):
        import numpy as np
        import torch
        import synthetic
        self.lib, self.T = lib, temperature
        M = rows_per_request * B
        self.M, V = M, shape["vocab"]
        m = rows_per_request - 1
        self.offs = [b * rows_per_request for b in range(B + 1)]
        self.model = lib.make_model(layers, head, shape["hidden"], shape["q_dim"], shape["inter"], V, shape["bits"])
        r = synthetic.rng(seed)
        self.h0 = torch.from_numpy(synthetic.activations(r, M, shape["hidden"]).view(np.int16)).cuda().view(
            torch.bfloat16)
        self.hidden = self.h0.clone()
        self.logits = torch.empty((M, V), dtype=torch.float32, device="cuda")
        self.out_len = torch.zeros(B, dtype=torch.int32, device="cuda")
        self.out_tokens = torch.zeros(M, dtype=torch.int32, device="cuda")
        self.ws = lib.workspace(lib.round_workspace_bytes(self.model, M))
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        nq = max(m * B, 1)
        self.q = torch.softmax(torch.randn((nq, V), generator=gen, device="cuda") * 2.0, dim=1)
        self.u = torch.cat([lib.philox_uniforms(seed, b, 0, rows_per_request) for b in range(B)])
        self.draft = torch.zeros(nq, dtype=torch.int32, device="cuda")
        # one eager greedy round to learn the target argmax, then drafts that agree with it w.p. 0.7
        self.run_eager(greedy=True)
        torch.cuda.synchronize()
        am = self.logits.argmax(dim=1).cpu().numpy()
        if m:
            d = [synthetic.agreeing_drafts(r, am[b * rows_per_request: b * rows_per_request + m], V, 0.7)
                 for b in range(B)]
            self.draft.copy_(torch.from_numpy(np.concatenate(d)))
        self.graph = None

    def run_eager(self, greedy=False, events=None):
        self.hidden.copy_(self.h0)
        self.lib.verify_round(self.model, self.offs, self.hidden, 0.0 if greedy else self.T, self.logits,
                              self.out_len, self.out_tokens, self.ws, q=self.q, draft=self.draft, u=self.u,
                              events=events)

    def capture(self):
        import torch
        self.run_eager()          # warm: kernel attributes are set outside capture
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(self.graph, stream=s):
                self.run_eager()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()


def max_over_ranks(v, dist=None, device="cuda"):
    """The largest of a per-rank value over all ranks (the slowest replica sets
    the job's time); v itself when there is no process group."""
    if not dist:
        return v
    import torch
    x = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(x, op=dist.ReduceOp.MAX)
    return float(x.item())


def time_replays(fn, steps, warmup, dist=None):
    """µs of each of `steps` back-to-back calls, CUDA events between them on the current stream."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record()
    for i in range(steps):
        fn()
        ev[i + 1].record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    return [ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(steps)]


def graph_of(fn):
    """fn's launches captured once into a CUDA graph (after one eager warm call),
    so that timing sees the device work and not the host's launch cost."""
    import torch
    fn()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def kernel_roofline(rnd, reps):
    """Dominant kernel: the persistent launch running every projection of a
    round.  Its duration comes from CUDA events the library records on the
    launching stream just before and after it.  Returns µs per launch (mean)."""
    import torch
    evs = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        e1.record()      # creates the underlying events
        evs.append((e0, e1))
    torch.cuda.synchronize()
    for e0, e1 in evs:
        rnd.run_eager(events=(e0, e1))
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in evs) * 1e3 / reps


def e2e_rounds(rnd, steps):
    """Host buffers in, host result out, through the public call: each step
    copies the round's inputs in from pinned host memory (the hidden rows on
    the round's stream; q, drafts and uniforms on a second stream after them,
    which the accept step waits for through accept_wait_event, so that copy
    overlaps the projections), runs the round, whose accept step writes
    out_len / out_tokens straight into pinned host memory, and waits for it;
    wall clock per round.  The copies and the round are one CUDA graph."""
    import torch
    host = [t.cpu().pin_memory() for t in (rnd.h0, rnd.q, rnd.draft, rnd.u)]
    len_host = torch.zeros_like(rnd.out_len, device="cpu").pin_memory()
    tok_host = torch.zeros_like(rnd.out_tokens, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = len_host.numel() * 4 + tok_host.numel() * 4
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    ready = torch.cuda.Event()

    def step():
        with torch.cuda.stream(main):
            rnd.hidden.copy_(host[0], non_blocking=True)
        side.wait_stream(main)   # after the hidden rows: one copy engine would otherwise queue them behind q
        with torch.cuda.stream(side):
            for dev, h in zip((rnd.q, rnd.draft, rnd.u), host[1:]):
                dev.copy_(h, non_blocking=True)
            ready.record(side)
        with torch.cuda.stream(main):
            rnd.lib.verify_round(rnd.model, rnd.offs, rnd.hidden, rnd.T, rnd.logits, len_host, tok_host,
                                 rnd.ws, q=rnd.q, draft=rnd.draft, u=rnd.u, stream=main, accept_wait=ready)

    main.wait_stream(torch.cuda.current_stream())
    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        with torch.cuda.stream(main):
            g.replay()
        main.synchronize()
    us = (time.perf_counter() - t0) * 1e6 / steps
    if not (0 < int(len_host[0]) <= rnd.out_tokens.numel()):
        raise SystemExit("end-to-end round left no result in host memory")
    return us, h2d, d2h


def device_model(lib, seed, shape, stats, packed=True):
    import torch
    from synthetic import model as _model
    layers, head = _model.device_random_model(seed, shape["n_layers"], shape["hidden"], shape["q_dim"],
                                              shape["kv_dim"], shape["inter"], shape["vocab"], shape["bits"], stats)
    if packed:      # one-time re-layout at load time, outside every timed region
        for w in [w for layer in layers for w in layer.values()] + [head]:
            w["packed"] = lib.pack(w)
        torch.cuda.synchronize()
    return layers, head


# ------------------------------------------------------------- workloads
def sweep_4b(lib, steps, warmup, hbm):
    """Qwen3-4B-shaped 4-bit round at every M = 1..32: µs per round, the knee,
    the cap the controller picks from the curve, and bf16 weights via cuBLAS."""
    import torch
    import synthetic
    from speculative_decoding_verify_qmm_gb300 import binding
    shape = SHAPE_4B
    layers, head = device_model(lib, 4321, shape, synthetic.LARGE_8BIT)
    wb = weight_bytes(shape)
    curve = {}
    for M in range(1, 33):
        rnd = Round(lib, layers, head, shape, M, 1, seed=500 + M, temperature=TEMPERATURE)
        rnd.capture()
        curve[M] = statistics.median(time_replays(rnd.replay, steps, warmup))
        del rnd
    t1 = curve[1]
    verify = [curve[M] for M in range(1, 33)]
    knee = binding.verify_knee(lib.lib, verify, 0.10)
    picks = {}
    for p in (0.5, 0.7, 0.9):
        c, rate = binding.best_cap(lib.lib, p, verify, [0.0] * 32, 0.0)
        picks[str(p)] = {"cap": c, "tokens_per_ms": round(rate * 1e3, 3)}
    # the same projections with unquantized bf16 weights (cuBLAS via torch), summed over a round:
    # two layer copies alternate so no projection's weights stay in L2 between calls
    h, dq, kv, i, v = (shape[k] for k in ("hidden", "q_dim", "kv_dim", "inter", "vocab"))
    dims = [(dq + 2 * kv, h), (h, dq), (2 * i, h), (h, i)]
    lay = [[torch.randn((n, k), device="cuda", dtype=torch.bfloat16) for n, k in dims] for _ in range(2)]
    hw = torch.randn((v, h), device="cuda", dtype=torch.bfloat16)
    bf16 = {}
    for M in (1, 2, 4, 8, 16, 32):
        xs = {k: torch.randn((M, k), device="cuda", dtype=torch.bfloat16) for _, k in dims}

        ys = {n: torch.empty((M, n), device="cuda", dtype=torch.bfloat16) for n, _ in dims}
        yh = torch.empty((M, v), device="cuda", dtype=torch.bfloat16)

        def layer_pair():
            for L in lay:
                for w in L:
                    torch.matmul(xs[w.shape[1]], w.t(), out=ys[w.shape[0]])
        g_pair = graph_of(layer_pair)
        g_head = graph_of(lambda: torch.matmul(xs[h], hw.t(), out=yh))
        t_pair = statistics.median(time_replays(g_pair.replay, max(10, steps // 2), warmup))
        t_head = statistics.median(time_replays(g_head.replay, max(10, steps // 2), warmup))
        bf16[str(M)] = round(t_pair / 2 * shape["n_layers"] + t_head, 1)
    del lay, hw
    out = {
        "workload": "Qwen3-4B-shaped verify round: 36 layers, hidden 2560, q 4096, kv 1024, inter 9728, 4-bit g64, "
                    "lm_head 2560->151936, T = 0.7, unit-packed weights",
        "weight_bytes_per_round": wb,
        "us_per_round": {str(M): round(t, 2) for M, t in curve.items()},
        "cost_ratio_vs_M1": {str(M): round(t / t1, 3) for M, t in curve.items()},
        "weight_stream_gbs": {str(M): round(wb / (t * 1e-6) / 1e9, 1) for M, t in curve.items()},
        "knee_width": knee, "knee_rule": "widest M with t(M) <= 1.10 t(1)",
        "cap_controller": {"picks": picks, "drafter_us": 0.0, "overhead_us": 0.0,
                           "note": "sv_best_cap on the measured t(M) curve; no drafter is built, so its cost is 0"},
        "bf16_weights_cublas_us_per_round": bf16,
        "bf16_note": "the same projections with bf16 weights (torch.matmul, cuBLAS, replayed from a CUDA graph), "
                     "summed to a round: a reference point for the quantized curve, not this library's path",
        "roofline": {"bound": "hbm", "achieved": round(wb / (curve[8] * 1e-6) / 1e9, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(wb / (curve[8] * 1e-6) / 1e9 / hbm, 3), "traffic": None,
                     "note": "whole round at M = 8 (weight bytes / replay time)"},
    }
    del layers, head
    torch.cuda.empty_cache()
    return out


def batched_27b(lib, steps, warmup, hbm):
    """27B-class 8-bit round: 64 layers, B = 4 requests x (1 + 7) rows, T = 1.0."""
    import torch
    import synthetic
    shape = SHAPE_27B
    layers, head = device_model(lib, 2727, shape, synthetic.LARGE_8BIT)
    wb = weight_bytes(shape)
    rnd = Round(lib, layers, head, shape, 8, 4, seed=2728, temperature=1.0)
    rnd.capture()
    sp = spread(time_replays(rnd.replay, max(steps, 50), warmup))
    kern = kernel_roofline(rnd, max(10, steps // 2))
    accepted = rnd.out_len.cpu().tolist()
    out = {
        "workload": "27B-class verify round: 64 layers, hidden 5120, q 6144, kv 1024, inter 17408, 8-bit g64, "
                    "lm_head 5120->151936, B = 4 requests x (1 + 7) rows = 32 rows, T = 1.0, per-request Philox",
        "weight_bytes_per_round": wb, "us_per_round": sp, "phases_per_launch": 4 * shape["n_layers"] + 1,
        "weight_stream_gbs": round(wb / (sp["median"] * 1e-6) / 1e9, 1),
        "pct_of_8tbs": round(100 * wb / (sp["median"] * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 1),
        "accepted_per_request_last_round": accepted,
        "roofline": {"bound": "hbm", "achieved": round(wb / (kern * 1e-6) / 1e9, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(wb / (kern * 1e-6) / 1e9 / hbm, 3), "traffic": None,
                     "kernel": "stream_kernel<8,4>: all 257 projections of the round", "us_per_launch": round(kern, 1)},
    }
    del rnd, layers, head
    torch.cuda.empty_cache()
    return out


# single projections of the one-layer 8B sweep and the tiny 4-bit layer:
# name -> (N, K, bits, the row counts timed)
PROJ_SHAPES = {"8b_" + name: (N, K, 8, (1, 2, 4, 6, 8, 12, 16, 17))
               for name, (N, K) in {"q": (4096, 4096), "k": (1024, 4096), "o": (4096, 4096),
                                    "gate": (12288, 4096), "down": (4096, 12288)}.items()}
PROJ_SHAPES["tiny_4bit_1024"] = (1024, 1024, 4, (1, 2, 4, 8))


def projections(lib, steps, warmup, hbm):
    """Single projections through sv_qmm_verify, rotating weight copies that
    together exceed 2 x L2, so every call streams its weights from HBM."""
    import numpy as np
    import torch
    import synthetic
    out = {}

    def run_shape(name, N, K, bits, stats, Ms, seed):
        per = N * K * (bits / 8 + 4 / 64)
        copies = max(2, int(np.ceil(2 * L2_BYTES / per)) + 1)
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        ws = [synthetic.device_quant_weight(gen, N, K, bits, stats) for _ in range(copies)]
        res = {}
        for M in Ms:
            x = torch.randn((M, K), device="cuda", dtype=torch.bfloat16)
            y = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
            wsp = lib.workspace(lib.qmm_workspace_bytes(M, N, K, bits))

            def calls():      # one call per weight copy, in turn
                for w in ws:
                    lib.qmm_verify(w["wq"], w["scales"], w["biases"], K, bits, x, y=y, workspace=wsp)
            g = graph_of(calls)
            t = statistics.median(time_replays(g.replay, max(10, steps // 2), warmup)) / copies
            res[str(M)] = {"us": round(t, 2), "gbs": round(per / (t * 1e-6) / 1e9, 1)}
        out[name] = {"N": N, "K": K, "bits": bits, "copies_rotated": copies, "by_M": res}
        del ws

    for name, (N, K, bits, Ms) in PROJ_SHAPES.items():
        stats = synthetic.LARGE_8BIT if bits == 8 else synthetic.TINY_4BIT
        run_shape(name, N, K, bits, stats, Ms, 60 + N + K if bits == 8 else 70)
    torch.cuda.empty_cache()
    return {"note": "µs per sv_qmm_verify call (activation preparation + matmul) within a CUDA graph that cycles "
                    "through the weight copies, median; GB/s = weight bytes / time",
            "peak_gbs": hbm, "shapes": out}


def wide(lib, steps, warmup, peaks):
    """tcgen05 matmul at M = 512 (a prefill-sized block) on 8B shapes."""
    import numpy as np
    import torch
    import synthetic
    tf_peak = peaks["bf16_tflops"] if peaks else 1900.0
    hbm = peaks["hbm_gbs"] if peaks else 6800.0
    out = {}
    for name, (N, K) in {"gate_up": (24576, 4096), "down": (4096, 12288), "q": (4096, 4096)}.items():
        M, bits = 512, 8
        per = N * K * (bits / 8 + 4 / 64)
        copies = max(2, int(np.ceil(2 * L2_BYTES / per)) + 1)
        gen = torch.Generator(device="cuda")
        gen.manual_seed(N + K)
        ws = [synthetic.device_quant_weight(gen, N, K, bits, synthetic.LARGE_8BIT) for _ in range(copies)]
        x = torch.randn((M, K), device="cuda", dtype=torch.bfloat16)
        y = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
        wsp = lib.workspace(lib.qmm_workspace_bytes(M, N, K, bits))

        def calls():          # one call per weight copy, in turn
            for w in ws:
                lib.qmm_verify(w["wq"], w["scales"], w["biases"], K, bits, x, y=y, workspace=wsp)
        g = graph_of(calls)
        t = statistics.median(time_replays(g.replay, max(10, steps // 2), warmup)) / copies
        tf = 2.0 * M * N * K / (t * 1e-6) / 1e12
        out[name] = {"N": N, "K": K, "M": M, "us": round(t, 2), "tflops": round(tf, 1),
                     "weight_gbs": round(per / (t * 1e-6) / 1e9, 1), "copies_rotated": copies}
        del ws
    # the gate|up shape across block widths: the tensor-memory kernel from 33 rows up, the
    # weight-streaming kernel at 32 for comparison
    N, K, bits = 24576, 4096, 8
    per = N * K * (bits / 8 + 4 / 64)
    copies = max(2, int(np.ceil(2 * L2_BYTES / per)) + 1)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(N + K + 1)
    ws = [synthetic.device_quant_weight(gen, N, K, bits, synthetic.LARGE_8BIT) for _ in range(copies)]
    by_m = {}
    for M in (32, 33, 64, 128, 256, 512):
        x = torch.randn((M, K), device="cuda", dtype=torch.bfloat16)
        y = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
        wsp = lib.workspace(lib.qmm_workspace_bytes(M, N, K, bits))

        def calls_m():
            for w in ws:
                lib.qmm_verify(w["wq"], w["scales"], w["biases"], K, bits, x, y=y, workspace=wsp)
        g = graph_of(calls_m)
        t = statistics.median(time_replays(g.replay, max(10, steps // 2), warmup)) / copies
        by_m[str(M)] = {"us": round(t, 2), "tflops": round(2.0 * M * N * K / (t * 1e-6) / 1e12, 1),
                        "weight_gbs": round(per / (t * 1e-6) / 1e9, 1)}
    del ws
    top = out["gate_up"]
    torch.cuda.empty_cache()
    return {"workload": "8-bit g64 projections at M = 512 rows through sv_qmm_verify (tcgen05.mma, fp16 operands, "
                        "fp32 accumulators in tensor memory)",
            "by_shape": out,
            "gate_up_by_M": by_m,
            "gate_up_by_M_note": "sv_qmm_verify on the 24576 x 4096 gate|up shape per block width; M = 32 runs the "
                                 "weight-streaming kernel, M >= 33 the tensor-memory kernel",
            "roofline": {"bound": "tensor", "achieved": top["tflops"], "peak": tf_peak, "unit": "TFLOP/s",
                         "frac": round(top["tflops"] / tf_peak, 3), "traffic": None,
                         "kernel": "wide_kernel<8> (gate_up 24576 x 4096, M = 512), whole call incl. preparation "
                                   "(CUDA-graph replay through the weight copies)",
                         "peak_source": "MEASURED_PEAKS.json bf16_tflops (burst; kind::f16 runs at the bf16 rate), "
                                        "of measured" if peaks else "fallback"},
            "hbm_peak_gbs": hbm}


def bits2_round(lib, steps, warmup, hbm):
    """The 27B-class round with 2-bit codes (the pages' 2-bit target, whose
    verify rows turn compute-bound early) at M = 1..8: us per round and the
    cost ratio against M = 1."""
    import torch
    import synthetic
    shape = dict(SHAPE_27B, bits=2)
    layers, head = device_model(lib, 2222, shape, synthetic.TINY_2BIT)
    wb = weight_bytes(shape)
    curve = {}
    for M in (1, 2, 3, 4, 6, 8):
        rnd = Round(lib, layers, head, shape, M, 1, seed=900 + M, temperature=TEMPERATURE)
        rnd.capture()
        curve[M] = statistics.median(time_replays(rnd.replay, steps, warmup))
        del rnd
    del layers, head
    torch.cuda.empty_cache()
    t1 = curve[1]
    return {"workload": "27B-class verify round with 2-bit g64 codes: 64 layers, hidden 5120, q 6144, kv 1024, "
                        "inter 17408, lm_head 5120->151936, T = 0.7, unit-packed weights",
            "weight_bytes_per_round": wb,
            "us_per_round": {str(k): round(v, 2) for k, v in curve.items()},
            "cost_ratio_vs_M1": {str(k): round(v / t1, 3) for k, v in curve.items()},
            "weight_stream_gbs": {str(k): round(wb / (v * 1e-6) / 1e9, 1) for k, v in curve.items()},
            "roofline": {"bound": "hbm", "achieved": round(wb / (t1 * 1e-6) / 1e9, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(wb / (t1 * 1e-6) / 1e9 / hbm, 3), "traffic": None,
                         "note": "whole round at M = 1 (weight bytes / replay time)"}}


def moe_gather(lib, steps, warmup, hbm):
    """Mixture-of-experts verify rows through sv_gather_qmm: 128 experts, each
    row routed to 8 of them (a 30B-A3B-class expert layer, gate|up 2 x 768 x
    2048, 4-bit).  Every extra verify row pulls in more experts: us per call
    and the distinct experts' bytes per call, over 16 route sets per width."""
    import numpy as np
    import torch
    import synthetic
    E, N, K, bits, top = 128, 2 * 768, 2048, 4, 8
    gen = torch.Generator(device="cuda")
    gen.manual_seed(3030)
    w = synthetic.device_quant_weight(gen, E * N, K, bits, synthetic.TINY_4BIT)
    per_expert = N * K * (bits / 8 + 4 / 64)
    r = synthetic.rng(3031)
    out = {}
    for M in (1, 2, 4, 8, 16):
        x = synthetic.device_activations(gen, M, K)
        sets, distinct = [], []
        for _ in range(16):
            rows = np.repeat(np.arange(M, dtype=np.int32), top)
            exps = np.concatenate([r.choice(E, top, replace=False) for _ in range(M)]).astype(np.int32)
            sets.append((torch.from_numpy(rows).cuda(), torch.from_numpy(exps).cuda()))
            distinct.append(len(set(exps.tolist())))
        P = M * top
        y = torch.empty((P, N), dtype=torch.bfloat16, device="cuda")
        wsp = lib.workspace(lib.lib.sv_gather_qmm_workspace_bytes(P, M, N, K, E, bits))

        def calls():
            for pr, pe in sets:
                lib.gather_qmm(w["wq"], w["scales"], w["biases"], E, K, bits, x, pr, pe, y=y, workspace=wsp)
        g = graph_of(calls)
        t = statistics.median(time_replays(g.replay, max(10, steps // 2), warmup)) / len(sets)
        eb = statistics.fmean(distinct) * per_expert
        out[str(M)] = {"us": round(t, 2), "distinct_experts": round(statistics.fmean(distinct), 1),
                       "expert_bytes": round(eb), "gbs": round(eb / (t * 1e-6) / 1e9, 1)}
    del w
    torch.cuda.empty_cache()
    top_m = out["16"]
    return {"workload": "gather-qmm over 128 stacked 4-bit g64 experts (gate|up 1536 x 2048 each), 8 experts per "
                        "row, M = 1..16 verify rows; 16 random route sets per width in one CUDA graph",
            "by_M": out,
            "roofline": {"bound": "hbm", "achieved": top_m["gbs"], "peak": hbm, "unit": "GB/s",
                         "frac": round(top_m["gbs"] / hbm, 3), "traffic": None,
                         "note": "M = 16: distinct selected experts' bytes / call time"}}


def accept_variants(lib, steps, warmup, hbm):
    """The accept step's f2 variants at the full vocabulary (V = 151936, m = 7,
    T = 0.8): lossless top-k / top-p truncated accept, the truncated draft
    probabilities, and log-probabilities with the top 5 from the logits."""
    import numpy as np
    import torch
    import synthetic
    r = synthetic.rng(4040)
    V, m, T = 151936, 7, 0.8
    z, q = synthetic.logits_and_draft_probs(r, m, V)
    draft = synthetic.sample_drafts(r, q)
    u = synthetic.accept_uniforms(r, m + 1)
    dz, dq = torch.from_numpy(z).cuda(), torch.from_numpy(q).cuda()
    dd, du = torch.from_numpy(draft).cuda(), torch.from_numpy(u).cuda()
    chosen = torch.from_numpy(np.argmax(z, axis=1).astype(np.int32)).cuda()
    ws = lib.workspace(lib.accept_workspace_bytes(1, m + 1))
    probs_out = torch.empty_like(dq)
    cases = {
        "accept_plain": (lambda: lib.spec_accept_truncated([0, m + 1], dz, dd, T, 0, 1.0, q=dq, u=du, workspace=ws),
                         (2 * m + 1) * V * 4),
        "accept_top_k_50_top_p_0.9": (lambda: lib.spec_accept_truncated([0, m + 1], dz, dd, T, 50, 0.9, q=dq, u=du,
                                                                          workspace=ws), (2 * m + 1) * V * 4),
        "truncate_probs_top_p_0.9": (lambda: lib.truncate_probs(dq, 0, 0.9, out=probs_out), 2 * m * V * 4),
        "logprobs_top5": (lambda: lib.logprobs(dz, T, chosen=chosen, top_n=5), (m + 1) * V * 4),
    }
    out = {}
    for name, (fn, nbytes) in cases.items():
        g = graph_of(fn)
        t = statistics.median(time_replays(g.replay, max(20, steps), warmup))
        out[name] = {"us": round(t, 2), "bytes_read": nbytes, "gbs": round(nbytes / (t * 1e-6) / 1e9, 1)}
    if lib.device_error():
        raise SystemExit("device error in the accept variants")
    return {"workload": "V = 151936, m = 7 drafts, T = 0.8, one request; each call replayed from a CUDA graph",
            "calls": out,
            "note": "latency-bound: a few passes over 8 rows of 608 KB from L2"}


# ---------------------------------------------------------- CPU oracle leg
SAMPLE_ROWS = 4096       # per projection in the round sample (about 1.5 s of all-core CPU work)
PROJ_SAMPLE_ROWS = 256   # per single projection, at each of its row counts


def oracle_sample(shape, M, temperature, seed=7):
    """One bounded sample of a verify round on the CPU oracle.

    SAMPLE_ROWS weight rows of each projection of one layer (q|k|v fed by the
    first RMSNorm, o, gate|up fed by the second, down fed by SwiGLU, with the
    residual adds) and of the vocab head, each part's time scaled by the
    rows it stands for in a round (rows in the projection / rows sampled,
    times the layer count), plus the accept step on the full-width rows.
    Returns (estimated µs per round, seconds spent)."""
    import numpy as np
    from oracle import accept as oa, chain, glue
    import synthetic
    r = synthetic.rng(seed)
    h, dq, kv, i, v = (shape[k] for k in ("hidden", "q_dim", "kv_dim", "inter", "vocab"))
    L, bits, stats = shape["n_layers"], shape["bits"], synthetic.LARGE_8BIT
    R = SAMPLE_ROWS
    parts = {"qkv": (dq + 2 * kv, h), "o": (h, dq), "gate_up": (2 * i, h), "down": (h, i), "head": (v, h)}
    w = {k: synthetic.quant_weight(r, R, K, bits, stats) for k, (N, K) in parts.items()}
    x_h = synthetic.activations(r, M, h)
    x_q = synthetic.activations(r, M, dq)
    x_i = synthetic.activations(r, M, i)
    z, q = synthetic.logits_and_draft_probs(r, M - 1, v)
    draft = synthetic.sample_drafts(r, q) if M > 1 else np.zeros(0, np.int32)
    u = synthetic.accept_uniforms(r, M)
    est, spent = 0.0, time.perf_counter()

    def timed(fn, scale):
        nonlocal est
        t0 = time.perf_counter()
        out = fn()
        est += (time.perf_counter() - t0) * scale
        return out
    # projections: the sampled rows stand for the projection's N rows in each of L layers
    timed(lambda: chain.project_normed(w["qkv"], x_h), parts["qkv"][0] / R * L)
    timed(lambda: chain.project(w["o"], x_q), parts["o"][0] / R * L)
    timed(lambda: chain.project_normed(w["gate_up"], x_h), parts["gate_up"][0] / R * L)
    s = timed(lambda: glue.swiglu(x_i, x_i), L)                 # glue on full rows, once per layer
    timed(lambda: chain.project(w["down"], s), parts["down"][0] / R * L)
    timed(lambda: (glue.residual_add(x_h, x_h), glue.residual_add(x_h, x_h)), L)
    timed(lambda: chain.normed_f64(w["head"], x_h), parts["head"][0] / R)
    timed(lambda: oa.spec_accept(z, q, draft, temperature, u), 1.0)
    return est * 1e6, time.perf_counter() - spent


def oracle_projection_sample(reps=3, seed=11):
    """The CPU oracle's qmm_verify on PROJ_SAMPLE_ROWS weight rows of each single
    projection, at every row count of PROJ_SHAPES, scaled to the projection's
    N rows: estimated µs per call (median of `reps`)."""
    import numpy as np
    from oracle import qmm as oq
    import synthetic
    r = synthetic.rng(seed)
    out = {}
    for name, (N, K, bits, Ms) in PROJ_SHAPES.items():
        stats = synthetic.LARGE_8BIT if bits == 8 else synthetic.TINY_4BIT
        R = min(PROJ_SAMPLE_ROWS, N)
        w = synthetic.quant_weight(r, R, K, bits, stats)
        res = {}
        for M in Ms:
            x = synthetic.activations(r, M, K)
            ts = []
            for _ in range(reps):
                t0 = time.perf_counter()
                oq.qmm_verify(w["wq"], w["scales"], w["biases"], K, bits, x)
                ts.append((time.perf_counter() - t0) * N / R)
            res[str(M)] = round(statistics.median(ts) * 1e6, 1)
        out[name] = res
    return out


SAMPLE_NOTE = ("%d weight rows of each projection of one layer (with the RMSNorm, SwiGLU and residual glue) and of "
               "the vocab head, each scaled by the rows it stands for in the round, plus the accept step on the "
               "full-width rows; extrapolated to one round" % SAMPLE_ROWS)


def cpu_sample_main(args):
    """--cpu-sample: run the oracle sample `reps` times in this process (the
    caller sets the BLAS thread count in the environment) and print a JSON line."""
    if args.cpu_proj:
        oracle_projection_sample(1)                         # warm
        print(json.dumps(oracle_projection_sample(args.reps)))
        return
    M = args.only_m or 8
    oracle_sample(SHAPE_8B, M, TEMPERATURE)                 # warm
    runs = [oracle_sample(SHAPE_8B, M, TEMPERATURE) for _ in range(args.reps)]
    us = [u for u, _ in runs]
    print(json.dumps({"us_median": statistics.median(us), "us_all": us, "seconds": sum(s for _, s in runs),
                      "threads": os.environ.get("OPENBLAS_NUM_THREADS", "default")}))


def cpu_baseline(M, reps):
    """The oracle sample on 1 core and on all cores of this host (child processes
    with the BLAS thread count set before numpy loads)."""
    out = {}
    ncpu = os.cpu_count() or 1
    # one timed sample on one core (several seconds), `reps` on all cores
    for label, threads, n in (("single_core", 1, 1), ("all_cores", ncpu, reps)):
        env = dict(os.environ, OPENBLAS_NUM_THREADS=str(threads), OMP_NUM_THREADS=str(threads),
                   MKL_NUM_THREADS=str(threads), CUDA_VISIBLE_DEVICES="")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", "--reps", str(n),
                            "--only-m", str(M)], env=env, capture_output=True, text=True, timeout=900)
        if r.returncode != 0:
            out[label] = {"error": r.stderr[-400:]}
            continue
        d = json.loads(r.stdout.strip().splitlines()[-1])
        out[label] = {"value": d["us_median"], "cores": threads, "cpu_seconds": round(d["seconds"], 2)}
    # single projections of the one-layer sweeps on one core, beside the GPU's `projections`
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", "--cpu-proj", "--reps", "3"],
                       env=env, capture_output=True, text=True, timeout=900)
    out["projections_single_core"] = (
        {"us_per_call": json.loads(r.stdout.strip().splitlines()[-1]), "cores": 1,
         "sample": "%d weight rows of each projection, scaled to its N rows; median of 3" % PROJ_SAMPLE_ROWS}
        if r.returncode == 0 else {"error": r.stderr[-400:]})
    return out


# --------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true", help="the headline round only (no other workloads)")
    ap.add_argument("--layers", type=int, default=SHAPE_8B["n_layers"],
                    help="fewer layers of the same shapes: a small case for profiler captures, not a bench line")
    ap.add_argument("--layout", default="packed", choices=["packed", "canonical"],
                    help="weights streamed from the unit-packed copy (sv_qmm_pack) or the canonical tensors")
    ap.add_argument("--only-m", type=int, default=0, help="time only this row count (default: 1, 8 and 16)")
    ap.add_argument("--cpu-sample", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--reps", type=int, default=3, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-proj", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_sample:
        return cpu_sample_main(args)
    assert args.warmup >= 3, "at least 3 warm-up steps"
    shape = dict(SHAPE_8B, n_layers=args.layers)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    M = args.only_m or 8
    wbytes = weight_bytes(shape)
    config = {"workload": "Qwen3-8B-shaped verify round: %d layers x (q|k|v, o, gate|up, down) 8-bit g64 + "
                          "lm_head 4096->151936 + spec_accept" % shape["n_layers"],
              "M": M, "m": M - 1, "temperature": TEMPERATURE, "draft_agreement": 0.7,
              "weight_bytes_per_round": wbytes, "l2": "no flush: %.2f GB of weights per round >> 129 MB L2" % (wbytes / 1e9),
              "parallelism": "replicas" if args.gpus > 1 else "single GPU"}

    if args.impl == "reference":
        if rank != 0:
            return
        for _ in range(args.warmup):
            oracle_sample(SHAPE_8B, M, TEMPERATURE)
        runs = [oracle_sample(SHAPE_8B, M, TEMPERATURE) for _ in range(args.steps)]
        us = statistics.median([u for u, _ in runs])
        spent = sum(s for _, s in runs)
        line = {"impl": "reference", "metric": METRIC, "value": us, "unit": "us/round", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64 (CPU oracle)", "data": "synthetic",
                "config": config,
                "extrapolated": True,
                "extrapolation": "each step times one bounded sample of a round on the CPU oracle (%s); value is "
                                 "the median estimate of a whole round, so steps x ms_per_step exceeds this run's "
                                 "wall time (%.1f s of sampled work)" % (SAMPLE_NOTE, spent),
                "cpu_baseline": {"value": us, "unit": "us/round", "cores": os.cpu_count(), "kind": "oracle",
                                 "sample": SAMPLE_NOTE, "cpu_seconds": round(spent, 2)},
                "e2e": {"value": us, "unit": "us/round", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    # the CPU baseline runs first, in child processes, before this process touches the GPU
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(M, 3)
        allc = cb.get("all_cores", {})
        cpu = {"value": allc.get("value"), "unit": "us/round", "cores": allc.get("cores"), "kind": "oracle",
               "sample": SAMPLE_NOTE, "single_core": cb.get("single_core"), "all_cores": allc,
               "rule": "the same sample as bench.py --impl reference",
               "projections_single_core": cb.get("projections_single_core")}
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verify_qmm_gb300 import binding
    import synthetic
    lib = binding.load()
    peaks = measured_peaks()
    hbm = peaks["hbm_gbs"] if peaks else 6800.0

    layers, head = device_model(lib, 1234 + rank, shape, synthetic.LARGE_8BIT, packed=args.layout == "packed")
    ms = (M,) if args.only_m else (1, 8, 16)
    rounds = {}
    for Mx in ms:
        rnd = Round(lib, layers, head, shape, Mx, 1, seed=77 + Mx, temperature=TEMPERATURE)
        rnd.capture()
        rounds[Mx] = rnd

    with ClockSampler(local) as clk:
        t = {}
        for Mx in ms:
            if Mx != M:
                t[Mx] = statistics.median(time_replays(rounds[Mx].replay, args.steps, args.warmup, dist))
        t[M] = statistics.median(time_replays(rounds[M].replay, args.steps, args.warmup, dist))
    clocks = clk.summary()
    err = lib.device_error()
    if err:
        raise SystemExit("device error word 0x%x after the timed rounds" % err)

    us = {k: max_over_ranks(v, dist) for k, v in t.items()}
    gbs = {k: wbytes / (v * 1e-6) / 1e9 for k, v in us.items()}
    spreads = {str(Mx): spread(time_replays(rounds[Mx].replay, 100, 3)) for Mx in ms}

    # dominant kernel: the persistent matmul launch of the round
    dur_us = kernel_roofline(rounds[M], max(10, args.steps // 2))
    achieved = wbytes / (dur_us * 1e-6) / 1e9
    e2e_us, h2d, d2h = e2e_rounds(rounds[M], max(10, args.steps // 2))
    del rounds, layers, head
    torch.cuda.empty_cache()

    extra = {}
    if not args.quick and world == 1 and args.layers == SHAPE_8B["n_layers"]:
        extra["sweep_4b"] = sweep_4b(lib, args.steps, args.warmup, hbm)
        extra["batched_27b"] = batched_27b(lib, args.steps, args.warmup, hbm)
        extra["projections"] = projections(lib, args.steps, args.warmup, hbm)
        extra["wide"] = wide(lib, args.steps, args.warmup, peaks)
        extra["bits2_27b"] = bits2_round(lib, args.steps, args.warmup, hbm)
        extra["moe_gather"] = moe_gather(lib, args.steps, args.warmup, hbm)
        extra["accept_variants"] = accept_variants(lib, args.steps, args.warmup, hbm)
        if lib.device_error():
            raise SystemExit("device error after the additional workloads")

    launches_per_round = 4  # input preparation, the projections, row-statistics merge, accept
    line = {
        "metric": METRIC, "value": us[M] / world, "unit": "us/round", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us[M] / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "q8 codes x bf16 activations (fp16 MMA), fp32 accumulate",
        "data": "synthetic (seeded random weights and activations of the stated shapes)", "config": config,
        "weight_layout": args.layout,
        "statistic": "median of the timed replays (per-replay CUDA events)",
        "us_per_round": {str(k): round(v, 2) for k, v in sorted(us.items())},
        "replay_spread_us": spreads,
        "weight_stream_gbs": {str(k): round(v, 1) for k, v in sorted(gbs.items())},
        "pct_of_measured_hbm": {str(k): round(100 * v / hbm, 1) for k, v in sorted(gbs.items())},
        "pct_of_8tbs": {str(k): round(100 * v / NOMINAL_HBM_GBS, 1) for k, v in sorted(gbs.items())},
        "cost_ratio_vs_M1": {str(k): round(us[k] / us[1], 3) for k in sorted(us)} if 1 in us else None,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 3), "traffic": measured_traffic(M, wbytes),
                     "traffic_unit": "bytes per launch (ncu dram read + write, scaled from the profiled case)",
                     "kernel": "stream_kernel<8,%d>: all %d projections of the M=%d round in one launch" % (
                         (M + 7) // 8, 4 * shape["n_layers"] + 1, M),
                     "us_per_launch": round(dur_us, 1), "bytes_per_launch": round(wbytes),
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (burst copy), of measured" if peaks
                     else "fallback 6.8 TB/s"},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_us, 2), "unit": "us/round", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_round * args.steps,
        "gpu_launches_note": "kernels per timed M=%d region (%d per round)" % (M, launches_per_round),
        "clocks": clocks,
    }
    line.update(extra)
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


# -------------------------------------------------------- ncu DRAM traffic
# DRAM bytes (read + write) per launch of the persistent kernel, from one ncu
# capture of a smaller round (4 layers, M = 8), scaled to a full launch by
# weight bytes; valid only for the kernel source it was taken on, so the
# source's hash is checked and the figure dropped when it differs.
TRAFFIC_CAPTURE = {"sha256": "4b3b66edbde812a15ac0db0a981d02a4295e53a7e036ca7ec8f645652dcfee63", "M": 8,
                   "bytes": 1481640192 + 7081728, "weight_bytes": 1481211904}


def measured_traffic(M, wbytes):
    import hashlib
    if not TRAFFIC_CAPTURE or TRAFFIC_CAPTURE["M"] != M:
        return None
    src = os.path.join(ROOT, "speculative_decoding_verify_qmm_gb300", "csrc", "stream_kernel.cuh")
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != TRAFFIC_CAPTURE["sha256"]:
        return None
    return round(TRAFFIC_CAPTURE["bytes"] * wbytes / TRAFFIC_CAPTURE["weight_bytes"])


if __name__ == "__main__":
    main()
