"""Benchmark of the QSA layer step on GB300.

Default workload: the fixed four-row verify at a 261,120-token context,
bf16 K/V and index keys (pooled keys fp32), 24 query heads over 2 KV heads,
head_dim 256, 12 independent QSA layers, top 512 blocks plus the tail.
One bench "step" is one pass of the whole hot path -- pool the block the new
rows completed and score every visible block (one launch), select the top 512, sparse
attention with its split merge -- over all 12 layers, layer after layer on
one stream, captured once in a CUDA graph.  The metric is QSA layer-steps/s.

Prints ONE JSON line (rank 0): layer-steps/s, the roofline of the step's
scoring launch (algorithmic bytes / isolated launch time against the
measured HBM copy bandwidth), the end-to-end rate through the public API
with host buffers, the oracle's rate on the host cores, and the SM clocks.
Other workloads: the 65,536-token decode, a 2,048-row prefill chunk, and the
decode and verify steps over fp8 or q8 K/V state.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--layers N] [--impl ours|reference] [--no-cpu-baseline]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import WORKLOADS, make_layer  # noqa: E402

METRIC = "QSA layer-steps/s at 261,120-ctx verify M=4; HBM GB/s as % of GB300 roofline"
UNIT = "layer-steps/s"
L2_BYTES = 129 * 2 ** 20
FEW_ROWS = 8                  # rows per sequence the streaming few-row scoring serves
NOMINAL_HBM_GBS = 8000.0      # the 8 TB/s HBM roofline the target fraction is stated against
DTYPE_NAMES = {torch.bfloat16: "bf16", torch.float32: "f32"}


# ---------------------------------------------------------------------- workload setup

class Layer:
    """Device-resident state of one QSA layer for one sequence."""

    def __init__(self, L, M, dtype, seed, layer, n_planted, head_dim, device, kv_state=None):
        import indexed_sparse_attention_gb300 as qsa
        x = make_layer(L=L, M=M, dtype=dtype, seed=seed, layer=layer, n_planted=n_planted, head_dim=head_dim,
                       device=device)
        self.x = x
        self.kv_state = kv_state
        self.pooled = torch.empty((qsa.n_pooled_slots(L), 128), dtype=torch.float32, device=device)
        first_new = (L - M) // 4
        if first_new:
            qsa.pool_index_keys(x.idxk, self.pooled, 0, first_new)    # state from earlier steps (untimed)
        if kv_state is None:
            seg = qsa.Segment(x.k, x.v, 0)
        else:
            # Quantized caches written from the bf16 draw by the library's
            # append of every token (untimed): codes and scale records.
            codes = torch.uint8 if kv_state == "fp8" else torch.int8
            rec = 2 if kv_state == "fp8" else 2 * head_dim // 32
            kc = torch.zeros(x.k.shape, dtype=codes, device=device)
            vc = torch.zeros_like(kc)
            sc = torch.zeros((x.k.shape[0], L, rec), dtype=torch.float16, device=device)
            seg = qsa.Segment(kc, vc, 0, kv_scale=sc)
            fill = qsa.Seq(L, L, self.pooled, [seg], idx_keys=x.idxk)
            qsa.append_tokens(fill, x.k.contiguous(), x.v.contiguous(), x.idxk.clone())
            torch.cuda.synchronize(device)
        self.seq = qsa.Seq(L, M, self.pooled, [seg], idx_keys=x.idxk)
        self.step = qsa.LayerStep([self.seq], x.q_idx, x.q, out_dtype=torch.float32)


def build_layers(spec, n_layers, device, seed=0):
    return [Layer(spec["L"], spec["M"], spec["dtype"], seed, l, spec["n_planted"], spec["head_dim"], device,
                  spec.get("kv_state"))
            for l in range(n_layers)]


def launches_per_layer(layer) -> int:
    st = layer.step
    x = layer.x
    # Pooling runs inside the few-row scoring launch (bf16 index queries, <= 4
    # rows) when the step pools and scores in one call; else its own launch.
    fused = st.idx_array is not None and x.M <= FEW_ROWS and x.q_idx.dtype == torch.bfloat16
    n = (0 if fused else len(st.pool_jobs)) + 1 + 1 + 1   # pool, score, select, attention
    if x.M > FEW_ROWS and x.q_idx.dtype == torch.bfloat16:
        n += 1                                   # scoring on the tensor cores: + the key-plane split
    ws_needed = st.ws.numel() > 16
    return n + (1 if ws_needed else 0)           # + split merge (several splits per row)


def algorithmic_bytes(layer) -> dict:
    """Bytes one layer-step must move: the pooled keys once, the index
    queries, the selected K/V rows of both KV heads (each row once per query
    row), the queries and the outputs; not the dense K/V left unread and not
    the scores intermediate."""
    x = layer.x
    L, M = x.L, x.M
    # K/V bytes per (KV head, token): both rows, plus their scale record for
    # quantized state.
    kv_es = x.k.element_size()
    D_ = x.q.shape[2]
    if layer.kv_state == "fp8":
        kv_tok = 2 * D_ + 4
    elif layer.kv_state == "q8":
        kv_tok = 2 * D_ + D_ // 8
    else:
        kv_tok = 2 * D_ * kv_es
    D, Hq, Hkv = x.q.shape[2], x.q.shape[1], x.k.shape[0]
    idx_es = x.idxk.element_size()
    nb_max = L // 4
    new_blocks = sum(n for *_, n in layer.step.pool_jobs)
    pool_b = new_blocks * (4 * 128 * idx_es + 128 * 4)
    # The pooled keys once and the index queries; the scores the launch
    # writes for the selection are an intermediate and are not counted.
    score_b = nb_max * 128 * 4 + x.q_idx.numel() * x.q_idx.element_size()
    rows = []
    for p in x.row_pos:
        nb = (p + 1) // 4
        rows.append(4 * min(512, nb) + (p + 1) % 4)
    attn_b = sum(rows) * Hkv * kv_tok + x.q.numel() * x.q.element_size() + M * Hq * (D * 4 + 4)
    return {"pool": pool_b, "score": score_b, "attn": attn_b, "total": pool_b + score_b + attn_b,
            "score_pooled_only": nb_max * 128 * 4}


# ---------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [p.strip() for p in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------- distributed plumbing

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_rate(units_per_rank: int, world: int, ms_max: float) -> float:
    """Units every rank processed, over the slowest rank's time (ms): the
    whole-job throughput of N weak-scaled replicas."""
    return units_per_rank * world / (ms_max / 1e3)


def max_over_ranks(x: float, world) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------- the CPU oracle leg

def oracle_layer_steps(layers_host, n_threads, budget_s):
    """Time the oracle on host copies: per layer-step, pool the new block(s),
    score all visible blocks, select, attend.  Returns (layer-steps, seconds)."""
    import oracle
    oracle.set_threads(n_threads)
    done, elapsed = 0, 0.0
    for h in layers_host:
        t0 = time.perf_counter()
        new = oracle.pool(h["idxk"], h["b0"], h["nb"] - h["b0"]) if h["nb"] > h["b0"] else None
        pooled = h["pooled_old"] if new is None else __import__("numpy").concatenate([h["pooled_old"], new])
        s = oracle.score(h["q_idx"], pooled, h["row_pos"])
        sel, cnt, _ = oracle.select(s, h["row_pos"])
        oracle.attn(h["q"], h["k"], h["v"], h["row_pos"], sel, cnt)
        elapsed += time.perf_counter() - t0
        done += 1
        if elapsed >= budget_s:
            break
    return done, elapsed


def host_layer(x, rows=None):
    """Host copies of one layer's inputs (``make_layer`` output) for the
    oracle; pooled keys of the blocks before this step are state (pooled here
    by the oracle, untimed).  ``rows`` restricts the step to a sample of query
    rows (rows are independent)."""
    import oracle
    idxk = x.idxk.cpu()
    b0 = (x.L - x.M) // 4
    q_idx, q, pos = x.q_idx.cpu(), x.q.cpu(), x.row_pos
    if rows is not None:
        q_idx, q, pos = q_idx[rows], q[rows], [pos[r] for r in rows]
    return {"idxk": idxk, "q_idx": q_idx, "q": q, "k": x.k.cpu(), "v": x.v.cpu(),
            "row_pos": pos, "b0": b0, "nb": x.L // 4, "pooled_old": oracle.pool(idxk, 0, b0)}


def cpu_baseline(layers, min_s=10.0, max_s=30.0, max_layers=3, max_rows=64):
    """The oracle on a bounded sample of the workload (about min_s .. max_s
    seconds of host work): whole layer-steps, cycling over up to max_layers
    layers, when a layer has few rows; else a sample of rows of one
    layer-step (first and last included), grown until it takes about min_s,
    timed and scaled linearly to all rows (rows are independent)."""
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    M = layers[0].x.M
    if M <= max_rows:
        hosts = [host_layer(l.x) for l in layers[:max_layers]]
        n, secs = 0, 0.0
        while secs < min_s:
            dn, ds = oracle_layer_steps(hosts, cores, max_s - secs)
            n, secs = n + dn, secs + ds
        return {"value": n / secs, "unit": UNIT, "cores": cores, "kind": "oracle",
                "sample": f"{n} layer-steps of the workload (pool new blocks, score all blocks, select, attention "
                          f"over all rows and heads), cycling over {len(hosts)} layers, in fp64 C with OpenMP, "
                          f"{secs:.1f} s"}
    n_rows = max_rows
    while True:
        rows = sorted(set([0, M - 1] + [int(i * (M - 1) / (n_rows - 1)) for i in range(n_rows)]))
        _, secs = oracle_layer_steps([host_layer(layers[0].x, rows)], cores, max_s)
        if secs >= min_s or len(rows) >= M:
            break
        n_rows = min(M, int(len(rows) * min_s / max(secs, 1e-3) * 1.1) + 1)
    full = secs * M / len(rows)
    return {"value": 1.0 / full, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{len(rows)} of the {M} rows of one layer-step in fp64 C with OpenMP ({secs:.1f} s), "
                      f"scaled linearly in rows to {full:.1f} s per layer-step"}


# ---------------------------------------------------------------------- main

def run_reference(args, spec, world, rank):
    """The reference arm: the fp64 CPU oracle, timed on the host cores."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    n_layers = min(args.layers or spec["layers"], 2)
    # Inputs drawn on the host: nothing of the CUDA library runs on this arm.
    hosts = [host_layer(make_layer(L=spec["L"], M=spec["M"], dtype=spec["dtype"], seed=0, layer=l,
                                   n_planted=spec["n_planted"], head_dim=spec["head_dim"], device="cpu"))
             for l in range(n_layers)]
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    for i in range(args.warmup):
        oracle_layer_steps([hosts[i % len(hosts)]], cores, 1e9)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_layer_steps([hosts[i % len(hosts)]], cores, 1e9)
    secs = time.perf_counter() - t0
    value = args.steps / secs
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload, "layer_steps_per_step": 1,
                                            "context": spec["L"], "rows": spec["M"]},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "one layer-step of the workload per step, fp64 C oracle with OpenMP"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="verify_m4_261k_bf16",
                    choices=["verify_m4_261k_bf16", "decode_m1_65k_bf16", "prefill_t2048_100k_bf16",
                             "verify_m8_261k_bf16",
                             "tiny_verify_f32", "verify_m4_261k_fp8", "decode_m1_65k_fp8", "verify_m4_261k_q8",
                             "decode_m1_65k_q8"])
    ap.add_argument("--layers", type=int, default=0, help="layers per step (default: the workload's 12)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel-reps", type=int, default=200)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    spec = WORKLOADS[args.workload]
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, spec, world, rank)
        barrier(world)
        return

    import indexed_sparse_attention_gb300 as qsa
    from indexed_sparse_attention_gb300 import build as qsa_build
    if rank == 0:
        qsa_build.build()
    barrier(world)
    qsa.lib()
    dev = torch.device("cuda", local)
    n_layers = args.layers or spec["layers"]
    layers = build_layers(spec, n_layers, dev, seed=rank)
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize()

    def step_all():
        for l in layers:
            l.step.run()

    # Eager warm-up (sets kernel attributes outside capture), then capture.
    with torch.cuda.stream(stream):
        step_all()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step_all()
    torch.cuda.synchronize()

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except (AttributeError, RuntimeError):
        gpu_id = str(local)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for _ in range(args.steps):
            graph.replay()
        t_end.record(stream)
    t_end.synchronize()
    torch.cuda.synchronize()
    ms = t_start.elapsed_time(t_end)
    # Keep the clocks sampler fed for >= 1 s of load when the timed region was short.
    with torch.cuda.stream(stream):
        while time.perf_counter() - wall0 < 1.2:
            for _ in range(50):
                graph.replay()
            torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    ms = max_over_ranks(ms, world)
    ms_per_step = ms / args.steps
    value = whole_job_rate(n_layers * args.steps, world, ms)

    # Each step kind on its own: a graph of its 12 back-to-back launches (one
    # per layer), timed live.  Scoring is the dominant kernel (the roofline
    # line); the others show where the rest of the step goes.
    def time_kind(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in layers:
                fn(l.step)
        with torch.cuda.stream(stream):
            for _ in range(5):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.kernel_reps):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        return 1e3 * e0.elapsed_time(e1) / (args.kernel_reps * n_layers)

    kernel_us = {"pool": time_kind(lambda st: st.pool()), "score": time_kind(lambda st: st.score()),
                 "pool_score": time_kind(lambda st: st.pool_score()),
                 "select": time_kind(lambda st: st.select()),
                 "score_select": time_kind(lambda st: st.score_select()), "attend": time_kind(lambda st: st.attend())}
    # The roofline kernel timed without overlap: programmatic dependent launch
    # lets a scoring launch start streaming while its predecessor runs, so in
    # a graph of back-to-back scoring launches neighbours overlap.  Here each
    # launch is followed by a one-element torch kernel (launched without the
    # attribute, so the next launch waits for it), and a graph of the
    # separators alone is subtracted.
    sep_t = torch.zeros(1, device=dev)

    def time_isolated(fn):
        def graph_of(with_kernel):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for l in layers:
                    if with_kernel:
                        fn(l.step)
                    sep_t.add_(1.0)
            return g

        ga, gb = graph_of(True), graph_of(False)
        out = []
        for g in (ga, gb):
            with torch.cuda.stream(stream):
                for _ in range(5):
                    g.replay()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(args.kernel_reps):
                    g.replay()
                e1.record(stream)
            e1.synchronize()
            out.append(1e3 * e0.elapsed_time(e1) / (args.kernel_reps * n_layers))
        return out[0] - out[1]

    # Few rows with bf16 index queries: the step pools inside its scoring
    # launch (qsa_pool_score_blocks), so that launch is the one timed.
    fused = layers[0].step.idx_array is not None and spec["M"] <= FEW_ROWS and spec["dtype"] == torch.bfloat16
    score_us = time_isolated(lambda st: st.pool_score() if fused else st.score())
    attn_us = time_isolated(lambda st: st.attend()) if spec["M"] > FEW_ROWS else None

    # End to end through the public API with host buffers: per step, the new
    # rows' q, index queries, K/V and index keys of every layer go host ->
    # device into the caches, the layer chain runs, outputs come back.
    M = spec["M"]
    L = spec["L"]
    # Per step, every layer's inputs -- q, index queries and the new rows'
    # K, V and index keys (contiguous, as a model produces them) -- arrive in
    # one pinned host buffer and cross in one copy; qsa_append_score_blocks
    # writes the new rows into the caches, pools the blocks they complete and
    # scores; every layer's out and lse come back in one copy.
    def packed(tensors):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, n

    per_layer = []
    for l in layers:
        x = l.x
        per_layer.append([x.q, x.q_idx, x.k[:, L - M:].contiguous(), x.v[:, L - M:].contiguous(),
                          x.idxk[L - M:].contiguous()])
    flat_in = [t for ts in per_layer for t in ts]
    in_offs, in_bytes = packed(flat_in)
    stage_d = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    stage_h = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()

    def view(buf, off, t):
        n = t.numel() * t.element_size()
        return buf[off:off + n].view(t.dtype).view(t.shape)

    for off, t in zip(in_offs, flat_in):
        view(stage_h, off, t).copy_(t.cpu())
    out_shapes = [(l.step.out, l.step.lse) for l in layers]
    flat_out = [t for pair in out_shapes for t in pair]
    out_offs, out_bytes = packed(flat_out)
    out_d = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
    out_h = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    e2e_layers = []
    for i, l in enumerate(layers):
        q_v, qi_v, k_v, v_v, idx_v = (view(stage_d, in_offs[5 * i + j], per_layer[i][j]) for j in range(5))
        st = qsa.LayerStep([l.seq], qi_v, q_v, out_dtype=torch.float32)
        st.out = view(out_d, out_offs[2 * i], l.step.out)
        st.lse = view(out_d, out_offs[2 * i + 1], l.step.lse)
        e2e_layers.append((st, [(k_v, v_v, idx_v)]))
    h2d = sum(t.numel() * t.element_size() for t in flat_in)
    d2h = sum(t.numel() * t.element_size() for t in flat_out)

    def e2e_step():
        stage_d.copy_(stage_h, non_blocking=True)
        for st, nt in e2e_layers:
            st.run(new_tokens=nt)
        out_h.copy_(out_d, non_blocking=True)

    # The step as an application would replay it: one CUDA graph holding the
    # pinned host -> device copies, the layer chain through the public API and
    # the device -> host copies (the library's calls are capturable).
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e_step()
    torch.cuda.synchronize()
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph, stream=stream):
        e2e_step()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e_graph.replay()
    torch.cuda.synchronize()
    e2e_steps = max(10, min(args.steps, 200))
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_graph.replay()
        e1.record(stream)
    e1.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = whole_job_rate(n_layers * e2e_steps, world, e2e_ms)

    ab = algorithmic_bytes(layers[0])
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        peak_gbs, peak_src = float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        peak_gbs, peak_src = 6800.0, "fallback"
    score_bytes = ab["score"] + (ab["pool"] if fused else 0)
    score_gbs = score_bytes / (score_us * 1e-6) / 1e9
    step_gbs = ab["total"] * n_layers / (ms_per_step * 1e-3) / 1e9

    def traffic_of(kernel):
        """DRAM bytes per launch from the committed ncu counters, if they were
        taken on the kernel revision built now."""
        try:
            t = json.load(open(os.path.join(ROOT, "profiles", "kernel_traffic.json")))
            for e in t.get("entries", []):
                if (e.get("kernel") == kernel and e.get("rev") == KERNEL_REVS[kernel]
                        and e.get("workload") == args.workload):
                    return e["dram_bytes_per_launch"]
        except (OSError, ValueError, KeyError):
            pass
        return None

    # The scoring kernel this call runs (the library's choice by rows per
    # sequence): the TMA ring for 2 to 4 rows, direct loads for 1 and 5 to 8.
    if 2 <= M <= 4:
        score_kernel = "score_tma_pool_kernel" if fused else "score_tma_kernel"
    elif M <= FEW_ROWS:
        score_kernel = "score_direct_kernel"
    else:
        score_kernel = "score_tc_kernel"

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(layers)

    roofline = {"kernel": "pool_score_blocks (steps 1 + 2, one launch)" if fused else "score_blocks",
                "bound": "hbm", "achieved": score_gbs, "peak": peak_gbs,
                "unit": "GB/s", "frac": score_gbs / peak_gbs, "frac_of_8tbs": score_gbs / NOMINAL_HBM_GBS,
                "traffic": traffic_of(score_kernel), "traffic_kernel": score_kernel,
                "peak_source": f"{peak_src} (hbm_gbs, burst)", "us_per_launch": score_us,
                "timing": "graph of 12 launches each followed by a one-element non-PDL kernel, minus a graph "
                          "of those kernels alone (no overlap with neighbours)",
                "algorithmic_bytes_per_launch": score_bytes}
    roofline_scoring = None
    if M > FEW_ROWS:
        # Many rows (prefill).  Scoring is a dense contraction on the tensor
        # cores: algorithmic flops 2 x rows x 4 heads x blocks x 128; the
        # kernel executes three times as many (three bf16 planes of the fp32
        # keys).
        flops = 2.0 * M * 4 * (L // 4) * 128
        try:
            peak_tf, tf_src = float(peaks["bf16_tflops"]), "measured (bf16_tflops, burst)"
        except (KeyError, ValueError, TypeError):
            peak_tf, tf_src = 1900.0, "fallback"
        achieved = flops / (score_us * 1e-6) / 1e12
        roofline_scoring = dict(roofline)
        roofline_scoring.update({"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                                 "frac": achieved / peak_tf, "traffic": traffic_of("score_tc_kernel"),
                                 "peak_source": tf_src,
                                 "algorithmic_flops_per_launch": flops, "executed_flops_per_launch": 3 * flops})
        roofline_scoring.pop("algorithmic_bytes_per_launch")
        # The dominant kernel is the gathered attention (tcgen05): every row
        # moves its selected K and V rows of both KV groups into the SMs.  Most
        # of those bytes come from L2 (rows overlap across the 2,048 queries),
        # so the DRAM traffic is well below the algorithmic bytes.
        attn_gbs = ab["attn"] / (attn_us * 1e-6) / 1e9
        roofline = {"kernel": "sparse_attn (tcgen05 path)", "bound": "hbm", "achieved": attn_gbs,
                    "peak": peak_gbs, "unit": "GB/s", "frac": attn_gbs / peak_gbs,
                    "frac_of_8tbs": attn_gbs / NOMINAL_HBM_GBS,
                    "traffic": traffic_of("attn_tc_kernel"), "peak_source": f"{peak_src} (hbm_gbs, burst)",
                    "us_per_launch": attn_us, "timing": roofline["timing"],
                    "algorithmic_bytes_per_launch": ab["attn"]}

    launches = sum(launches_per_layer(l) for l in layers) * args.steps
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE_NAMES[spec["dtype"]], "data": "synthetic",
        "config": {"workload": args.workload, "context": L, "rows": M, "layers_per_step": n_layers,
                   "q_heads": layers[0].x.q.shape[1], "kv_heads": layers[0].x.k.shape[0],
                   "head_dim": layers[0].x.q.shape[2], "top_k_blocks": 512,
                   "kv_state": spec.get("kv_state") or "bf16",
                   "index_heads": 4, "index_dim": 128, "graph": "one CUDA graph per step (all layers)",
                   "l2": f"inputs larger than L2: {n_layers} distinct layers, "
                         f"{ab['total'] * n_layers / 2**20:.0f} MiB algorithmic bytes per step",
                   "parallelism": f"replicas x{world}"},
        "us_per_layer_step": 1e3 * ms_per_step / n_layers,
        "algorithmic_bytes_per_layer_step": ab["total"],
        "step_hbm_gbs": step_gbs,
        "step_frac_of_peak": step_gbs / peak_gbs,
        "step_frac_of_8tbs": step_gbs / NOMINAL_HBM_GBS,
        "roofline": roofline,
        **({"roofline_scoring": roofline_scoring} if roofline_scoring else {}),
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "mode": "one CUDA graph per step: one pinned host->device copy of every layer's q, index "
                        "queries and new K/V/index-key rows, per layer qsa_append_score_blocks (cache write, "
                        "pooling and scoring, one launch on the few-row path), selection and attention through "
                        "LayerStep (the C ABI), one device->host copy of every layer's out and lse"},
        "gpu_launches": launches,
        "us_per_launch_by_step": kernel_us,
        "clocks": {k: clk.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# Revision tags of the kernels as built now; DRAM counters in
# profiles/kernel_traffic.json count only for the revision they were taken on.
KERNEL_REVS = {"score_tma_kernel": "score_tma_2cta_bal_v1", "score_tma_pool_kernel": "score_tma_pool_2cta_bal_v1",
               "score_direct_kernel": "score_direct_v1",
               "attn_tc_kernel": "attn_tc_ring3_v1", "score_tc_kernel": "score_tc_planes3_v1"}

if __name__ == "__main__":
    main()
