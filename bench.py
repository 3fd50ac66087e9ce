"""Benchmark: one speculative-decoding verify round on a Qwen3-8B-shaped 8-bit target.

A step is one whole verify round: 36 layers of q|k|v, o, gate|up and down
projections (8-bit, group 64) with the RMSNorm / residual / SwiGLU steps fused
into the activation preparation, the 151936-row vocab head with its row
statistics, and the accept step (T = 0.7, drafts and draft probabilities
given).  The round is captured once into a CUDA graph and replayed.

Headline: microseconds per verify round at M = 8 rows (anchor + 7 drafts);
the same run also times M = 1 and M = 16 and reports the weight-stream
bandwidth (algorithmic weight bytes per round / round time) against the
measured HBM copy bandwidth.  All weights (8.04 GB) are far larger than L2,
so no flush is needed between rounds.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
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
SHAPE = dict(hidden=4096, q_dim=4096, kv_dim=1024, inter=12288, vocab=151936, n_layers=36, bits=8)
TEMPERATURE = 0.7
NOMINAL_HBM_GBS = 8000.0


def weight_bytes(shape):
    h, dq, kv, i, v, L, bits = (shape[k] for k in ("hidden", "q_dim", "kv_dim", "inter", "vocab", "n_layers", "bits"))
    per_weight = bits / 8 + 4 / 64
    layer = (dq + 2 * kv) * h + h * dq + 2 * i * h + h * i
    return (L * layer + v * h) * per_weight


def projection_list(shape):
    """(name, N, K) of every matmul launch of one round, in order."""
    h, dq, kv, i, v = (shape[k] for k in ("hidden", "q_dim", "kv_dim", "inter", "vocab"))
    per_layer = [("qkv", dq + 2 * kv, h), ("o", h, dq), ("gate_up", 2 * i, h), ("down", h, i)]
    return per_layer * shape["n_layers"] + [("lm_head", v, h)]


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


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
    """Device model, buffers and the captured graph of one verify round at M rows."""

    def __init__(self, lib, layers, head, shape, M, seed):
        import numpy as np
        import torch
        import synthetic
        self.lib, self.M = lib, M
        V = shape["vocab"]
        m = M - 1
        self.model = lib.make_model(layers, head, shape["hidden"], shape["q_dim"], shape["inter"], V, shape["bits"])
        r = synthetic.rng(seed)
        self.h0 = torch.from_numpy(synthetic.activations(r, M, shape["hidden"]).view(np.int16)).cuda().view(
            torch.bfloat16)
        self.hidden = self.h0.clone()
        self.logits = torch.empty((M, V), dtype=torch.float32, device="cuda")
        self.out_len = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.out_tokens = torch.zeros(M, dtype=torch.int32, device="cuda")
        self.ws = lib.workspace(lib.round_workspace_bytes(self.model, M))
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        self.q = torch.softmax(torch.randn((max(m, 1), V), generator=gen, device="cuda") * 2.0, dim=1)
        self.u = lib.philox_uniforms(seed, 0, 0, M)
        self.draft = torch.zeros(max(m, 1), dtype=torch.int32, device="cuda")
        self.offs = [0, M]
        # one eager round to learn the target argmax, then drafts that agree with it w.p. 0.7
        self.run_eager(greedy=True)
        torch.cuda.synchronize()
        am = self.logits.argmax(dim=1).cpu().numpy()
        if m:
            self.draft.copy_(torch.from_numpy(synthetic.agreeing_drafts(r, am[:m], V, 0.7)))
        self.graph = None

    def run_eager(self, greedy=False, events=None):
        self.hidden.copy_(self.h0)
        self.lib.verify_round(self.model, self.offs, self.hidden, 0.0 if greedy else TEMPERATURE, self.logits,
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


def time_rounds(rnd, steps, warmup, dist=None):
    import torch
    for _ in range(warmup):
        rnd.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        rnd.replay()
    e1.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    return e0.elapsed_time(e1) * 1e3 / steps     # us per round


def matmul_kernel_roofline(rnd, reps):
    """Dominant kernel: the persistent launch that runs all 4 * layers + 1
    projections of a round.  Its duration comes from CUDA events the library
    records on the launching stream just before and after it; the algorithmic
    bytes are the round's weight bytes.  Returns mean seconds per launch."""
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
    return sum(e0.elapsed_time(e1) for e0, e1 in evs) * 1e-3 / reps


def e2e_rounds(lib, rnd, steps):
    """Host buffers in, host result out: pinned H2D of the round's inputs, the
    round, D2H of out_len/out_tokens, each step; wall clock per round."""
    import torch
    h0_host = rnd.h0.cpu().pin_memory()
    q_host = rnd.q.cpu().pin_memory()
    d_host = rnd.draft.cpu().pin_memory()
    u_host = rnd.u.cpu().pin_memory()
    len_host = torch.zeros(1, dtype=torch.int32).pin_memory()
    tok_host = torch.zeros(rnd.M, dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h0_host, q_host, d_host, u_host))
    d2h = len_host.numel() * 4 + tok_host.numel() * 4
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        rnd.h0.copy_(h0_host, non_blocking=True)
        rnd.q.copy_(q_host, non_blocking=True)
        rnd.draft.copy_(d_host, non_blocking=True)
        rnd.u.copy_(u_host, non_blocking=True)
        rnd.replay()
        len_host.copy_(rnd.out_len, non_blocking=True)
        tok_host.copy_(rnd.out_tokens, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    us = (time.perf_counter() - t0) * 1e6 / steps
    return us, h2d, d2h


# ---------------------------------------------------------- CPU oracle leg
def oracle_round_sample(shape, M, seed=7):
    """Time the CPU oracle on a bounded sample of one round at M rows: one full
    layer (all seven projections and the glue), the vocab head on 8192 rows, and
    the accept step on the full-width logits rows; scaled to a whole round."""
    import numpy as np
    from oracle import accept as oa, chain, glue, qmm as oq
    import synthetic
    r = synthetic.rng(seed)
    h, dq, kv, i, v = (shape[k] for k in ("hidden", "q_dim", "kv_dim", "inter", "vocab"))
    bits, stats = shape["bits"], synthetic.LARGE_8BIT
    lay = {"q": synthetic.quant_weight(r, dq, h, bits, stats), "k": synthetic.quant_weight(r, kv, h, bits, stats),
           "v": synthetic.quant_weight(r, kv, h, bits, stats), "o": synthetic.quant_weight(r, h, dq, bits, stats),
           "gate": synthetic.quant_weight(r, i, h, bits, stats), "up": synthetic.quant_weight(r, i, h, bits, stats),
           "down": synthetic.quant_weight(r, h, i, bits, stats)}
    head_rows = 8192
    head = synthetic.quant_weight(r, head_rows, h, bits, stats)
    x = synthetic.activations(r, M, h)
    z, q = synthetic.logits_and_draft_probs(r, M - 1, v)
    draft = synthetic.sample_drafts(r, q) if M > 1 else np.zeros(0, np.int32)
    u = synthetic.accept_uniforms(r, M)
    t0 = time.perf_counter()
    hid = chain.layer_forward(x, lay)
    t1 = time.perf_counter()
    oq.lm_head_verify(head["wq"], head["scales"], head["biases"], h, bits, glue.rmsnorm(hid), TEMPERATURE)
    t2 = time.perf_counter()
    oa.spec_accept(z, q, draft, TEMPERATURE, u)
    t3 = time.perf_counter()
    est = shape["n_layers"] * (t1 - t0) + (t2 - t1) * v / head_rows + (t3 - t2)
    return est * 1e6, t3 - t0, "1 of %d layers + %d of %d vocab rows + accept, M=%d, scaled to a round" % (
        shape["n_layers"], head_rows, v, M)


_STEP_CACHE = {}


def oracle_step_sample(shape, M):
    """1024 gate rows (K = hidden) with the RMSNorm feeding them, per step, scaled to a whole round by weight bytes.

    Returns (estimated us per round, seconds spent)."""
    from oracle import glue, qmm as oq
    import synthetic
    if "w" not in _STEP_CACHE:
        r = synthetic.rng(11)
        _STEP_CACHE["w"] = synthetic.quant_weight(r, 1024, shape["hidden"], shape["bits"], synthetic.LARGE_8BIT)
        _STEP_CACHE["x"] = synthetic.activations(r, M, shape["hidden"])
    w, x = _STEP_CACHE["w"], _STEP_CACHE["x"]
    t0 = time.perf_counter()
    oq.qmm_verify(w["wq"], w["scales"], w["biases"], shape["hidden"], shape["bits"], glue.rmsnorm(x))
    secs = time.perf_counter() - t0
    sample_bytes = 1024 * shape["hidden"] * (shape["bits"] / 8 + 4 / 64)
    return secs * 1e6 * weight_bytes(shape) / sample_bytes, secs


def cpu_cores():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    try:
        from threadpoolctl import threadpool_info
        n = [p.get("num_threads", 0) for p in threadpool_info() if p.get("user_api") == "blas"]
        if n:
            return max(n)
    except ImportError:
        pass
    return os.cpu_count()


# -------------------------------------------------------- ncu DRAM traffic
# DRAM bytes (read + write) per launch of the persistent kernel, from one ncu
# capture of a smaller round (4 layers, M = 8), scaled to
# a full launch by weight bytes; valid only for the kernel source it was taken
# on, so the source's hash is checked and the figure dropped when it differs.
TRAFFIC_CAPTURE = {"sha256": "0f292be305e8bd4d84ab514826071a6eedc221f1a39c5abd086ee7d7e9034684", "M": 8,
                   "bytes": 1481508352 + 6188544, "weight_bytes": 1481211904}


def measured_traffic(M, wbytes):
    import hashlib
    if not TRAFFIC_CAPTURE or TRAFFIC_CAPTURE["M"] != M:
        return None
    src = os.path.join(ROOT, "speculative_decoding_verify_qmm_gb300", "csrc", "stream_kernel.cuh")
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != TRAFFIC_CAPTURE["sha256"]:
        return None
    return round(TRAFFIC_CAPTURE["bytes"] * wbytes / TRAFFIC_CAPTURE["weight_bytes"])


# --------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=SHAPE["n_layers"],
                    help="fewer layers of the same shapes: a small case for profiler captures, not a bench line")
    ap.add_argument("--layout", default="packed", choices=["packed", "canonical"],
                    help="weights streamed from the unit-packed copy (sv_qmm_pack) or the canonical tensors")
    ap.add_argument("--only-m", type=int, default=0, help="time only this row count (default: 1, 8 and 16)")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    shape = dict(SHAPE, n_layers=args.layers)

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
            oracle_step_sample(SHAPE, M)
        us_list = [oracle_step_sample(SHAPE, M)[0] for _ in range(args.steps)]
        us = statistics.median(us_list)
        sample = oracle_step_sample.__doc__.split("\n")[0]
        line = {"impl": "reference", "metric": METRIC, "value": us, "unit": "us/round", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64 (CPU oracle)", "data": "synthetic",
                "config": config,
                "cpu_baseline": {"value": us, "unit": "us/round", "cores": cpu_cores(), "kind": "oracle",
                                 "sample": sample},
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
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verify_qmm_gb300 import binding
    from synthetic import model as _model
    import synthetic
    lib = binding.load()

    layers, head = _model.device_random_model(1234 + rank, shape["n_layers"], shape["hidden"], shape["q_dim"],
                                              shape["kv_dim"], shape["inter"], shape["vocab"], shape["bits"],
                                              synthetic.LARGE_8BIT)
    if args.layout == "packed":      # one-time re-layout at load time, outside every timed region
        for w in [w for layer in layers for w in layer.values()] + [head]:
            w["packed"] = lib.pack(w)
        torch.cuda.synchronize()
    ms = (M,) if args.only_m else (1, 8, 16)
    rounds = {}
    for Mx in ms:
        rnd = Round(lib, layers, head, shape, Mx, seed=77 + Mx)
        rnd.capture()
        rounds[Mx] = rnd

    with ClockSampler(local) as clk:
        t = {}
        for Mx in ms:
            if Mx != M:
                t[Mx] = time_rounds(rounds[Mx], args.steps, args.warmup, dist)
        t[M] = time_rounds(rounds[M], args.steps, args.warmup, dist)
    clocks = clk.summary()
    err = lib.device_error()
    if err:
        raise SystemExit("device error word 0x%x after the timed rounds" % err)

    def max_over_ranks(v):
        if not dist:
            return v
        x = torch.tensor([v], dtype=torch.float64, device="cuda")
        dist.all_reduce(x, op=dist.ReduceOp.MAX)
        return float(x.item())

    us = {k: max_over_ranks(v) for k, v in t.items()}
    peaks = measured_peaks()
    hbm = peaks["hbm_gbs"] if peaks else 6800.0
    gbs = {k: wbytes / (v * 1e-6) / 1e9 for k, v in us.items()}

    # dominant kernel: the persistent matmul launch of the round
    dur_s = matmul_kernel_roofline(rounds[M], max(10, args.steps // 2))
    achieved = wbytes / dur_s / 1e9
    e2e_us, h2d, d2h = e2e_rounds(lib, rounds[M], max(10, args.steps // 2))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        est, secs, sample = oracle_round_sample(shape, M)
        cpu = {"value": est, "unit": "us/round", "cores": cpu_cores(), "kind": "oracle", "sample": sample,
               "cpu_seconds": secs}

    traffic = measured_traffic(M, wbytes)
    launches_per_round = 4  # input preparation, the projections, row-statistics merge, accept
    line = {
        "metric": METRIC, "value": us[M] / world, "unit": "us/round", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us[M] / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "q8 codes x bf16 activations (fp16 MMA), fp32 accumulate",
        "data": "synthetic (seeded random weights and activations of the stated shapes)", "config": config,
        "weight_layout": args.layout,
        "us_per_round": {str(k): round(v, 2) for k, v in sorted(us.items())},
        "weight_stream_gbs": {str(k): round(v, 1) for k, v in sorted(gbs.items())},
        "pct_of_measured_hbm": {str(k): round(100 * v / hbm, 1) for k, v in sorted(gbs.items())},
        "pct_of_8tbs": {str(k): round(100 * v / NOMINAL_HBM_GBS, 1) for k, v in sorted(gbs.items())},
        "cost_ratio_vs_M1": {str(k): round(us[k] / us[1], 3) for k in sorted(us)} if 1 in us else None,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 3), "traffic": traffic,
                     "traffic_unit": "bytes per launch (ncu dram read + write, scaled from the profiled case)",
                     "kernel": "stream_kernel<8,%d>: all %d projections of the M=%d round in one launch" % (
                         (M + 7) // 8, 4 * shape["n_layers"] + 1, M),
                     "us_per_launch": round(dur_s * 1e6, 1), "bytes_per_launch": round(wbytes),
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (burst copy), of measured" if peaks
                     else "fallback 6.8 TB/s"},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_us, 2), "unit": "us/round", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_round * args.steps,
        "gpu_launches_note": "kernels per timed M=%d region (%d per round)" % (M, launches_per_round),
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
