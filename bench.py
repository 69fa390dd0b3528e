"""Benchmark of the fused decode attention block on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--cluster-size C] [--batch-tile B]
                    [--stage-bytes S] [--ctas-per-sm X] [--no-graph]

One step = one decode attention-block call (RMSNorm, QKV, RoPE, KV append,
split-KV attention, O projection + residual) over one batch of synthetic
inputs; for the 32-layer long-context workload one step is the 32-layer
chain.  Inputs live in HBM before timing starts; between steps the next of R
independently seeded replicas is used, with R chosen so the replicas span at
least 4x the L2 size (L2 never serves a step's weights or KV).

Prints ONE JSON line (rank 0).  ``value`` is the achieved HBM throughput in
GB/s (algorithmic bytes of all ranks' steps / max-over-ranks time);
``us_per_step`` is the step latency.  N > 1 runs independent replicas, one
per GPU (the path has no cross-GPU exchange).
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

METRIC = "decode attention-block µs/step and achieved HBM GB/s (fraction of GB300 peak)"
# The largest single-GPU workload: the Llama-2-7B-shaped layer at 16384 cached
# positions, 32 independently seeded layers chained in one CUDA graph.
DEFAULT_WORKLOAD = "llama2_7b_layer_b1_p16384_f16_x32"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_L2_BYTES = 129 * 1024 * 1024
# The fused kernel's name by launch mode (cf_launch_info.mode): 0 the
# sequence-split kernel, 1 the batched row-split kernel.
KERNEL_NAMES = {0: "cf_decode_kernel", 1: "cf_rows_kernel"}


# ------------------------------------------------------------ host helpers --
def algorithmic_bytes(w, positions) -> int:
    """Bytes one decode step must move at minimum: weights, ln_weight, the KV
    read over positions [0, p_b) of every row, the new K/V written, hidden
    read, out written, positions read."""
    es = 4 if w.dtype == "f32" else 2
    d, nq, nkv, H, B = w.head_dim, w.n_q_heads, w.n_kv_heads, w.hidden, w.batch
    weights = H * w.qkv_cols * es + nq * d * H * es + H * es
    kv_read = sum(2 * int(p) * nkv * d * es for p in positions)
    kv_write = 2 * B * nkv * d * es
    io = 2 * B * H * es + 4 * B
    return weights + kv_read + kv_write + io


def ffn_bytes(wf) -> int:
    """Bytes the FFN after the attention block must move: W_gate, W_up, W_down,
    its norm weight, the rows read and written."""
    es = 4 if wf.dtype == "f32" else 2
    return 3 * wf.intermediate * wf.hidden * es + wf.hidden * es + 2 * wf.batch * wf.hidden * es


def ffn_flops(wf) -> int:
    return 6 * wf.batch * wf.intermediate * wf.hidden


def tensor_bytes(d) -> int:
    """Bytes of the tensors in a (possibly nested) dict of tensors."""
    return sum(tensor_bytes(v) if isinstance(v, dict) else v.numel() * v.element_size()
               for v in d.values())


def to_cpu(d):
    return {k: (to_cpu(v) if isinstance(v, dict) else v.cpu()) for k, v in d.items()}


def flops_per_step(w, positions) -> int:
    d, nq, H, B = w.head_dim, w.n_q_heads, w.hidden, w.batch
    proj = 2 * B * H * w.qkv_cols + 2 * B * nq * d * H
    attn = sum(4 * (int(p) + 1) * nq * d for p in positions)
    return proj + attn


def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            v = float(json.load(fh)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Translation units of the fused decode kernels and their launch planning; the
# hash covers them and every header they include (found by following the
# #include "..." lines), so a change to any of them invalidates a recorded
# ncu traffic figure.
FUSED_KERNEL_ROOTS = ("cf_api.cu", "cf_inst_bf16.cu", "cf_inst_f16.cu", "cf_inst_f32.cu",
                      "cf_inst_rows.cu", "cf_inst_rows_sweep.cu")
# The MLA variant's translation unit.
MLA_KERNEL_ROOTS = ("cf_mla.cu",)


def fused_kernel_sources(roots=FUSED_KERNEL_ROOTS) -> list[str]:
    import re
    dirs = [os.path.join(ROOT, "attention_block_gb300", "csrc"), os.path.join(ROOT, "include")]
    seen, todo = {}, list(roots)
    while todo:
        name = todo.pop()
        if name in seen:
            continue
        for d in dirs:
            path = os.path.join(d, name)
            if os.path.exists(path):
                seen[name] = path
                with open(path, encoding="utf-8") as fh:
                    todo += re.findall(r'^\s*#\s*include\s+"([^"]+)"', fh.read(), re.M)
                break
    return [seen[n] for n in sorted(seen)]


def kernel_source_hash(roots=FUSED_KERNEL_ROOTS) -> str:
    h = hashlib.sha256()
    for path in fused_kernel_sources(roots):
        with open(path, "rb") as fh:
            h.update(os.path.basename(path).encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, roots=FUSED_KERNEL_ROOTS):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)
        ent = rec.get(workload)
        if ent and ent.get("kernel_src_sha") == kernel_source_hash(roots):
            return int(ent["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def parse_clocks(lines):
    """Parse nvidia-smi CSV samples -> clocks dict for the JSON line."""
    sm, mx, reasons, loaded = [], 0.0, set(), []
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 9 or not parts[1].split()[0].replace(".", "").isdigit():
            continue
        try:
            cur = float(parts[1].split()[0])
            mx = max(mx, float(parts[2].split()[0]))
            pw = float(parts[3].split()[0])
        except ValueError:
            continue
        sm.append(cur)
        loaded.append((cur, pw))
        for name, val in zip(names, parts[5:9]):
            if val.lower() == "active":
                reasons.add(name)
    under = [c for c, p in loaded if p > 200.0] or sm
    return {"sm_mhz": statistics.median(under) if under else None,
            "sm_max_mhz": mx or None, "reasons": sorted(reasons), "samples": len(sm)}


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        self.stamped = []      # (host time, line)
        self.window = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()
            while not self.stamped and time.time() - t0 < 10.0:
                time.sleep(0.01)  # first sample in hand before timing starts
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.stamped.append((time.time(), ln))

    def mark(self, t_begin: float, t_end: float):
        """Host times bracketing the timed region."""
        self.window = (t_begin, t_end)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)
        return False

    def result(self):
        """Samples inside the timed window; if the window is shorter than the
        sampling period, the samples just before and after it (flagged)."""
        if self.window is None:
            return parse_clocks([ln for _, ln in self.stamped])
        a, b = self.window
        inside = [ln for t, ln in self.stamped if a <= t <= b]
        if inside:
            res = parse_clocks(inside)
            res["window"] = "timed region"
            return res
        before = [ln for t, ln in self.stamped if t < a][-2:]
        after = [ln for t, ln in self.stamped if t > b][:2]
        res = parse_clocks(before + after)
        res["window"] = "samples bracketing a timed region shorter than the sampling period"
        return res


def allgather_rows(mine, world: int, device):
    """All ranks' float rows (one list per rank), via torch.distributed."""
    import torch
    import torch.distributed as dist
    if world == 1:
        return [list(mine)]
    t = torch.tensor([list(mine)], dtype=torch.float64, device=device)
    gathered = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(gathered, t)
    return [g[0].tolist() for g in gathered]


def aggregate(per_rank):
    """Combine per-rank (bytes, seconds, steps) -> whole-job numbers: total
    bytes over the max time (the slowest rank bounds the job)."""
    tot_bytes = sum(r[0] for r in per_rank)
    t = max(r[1] for r in per_rank)
    return {"gbs": tot_bytes / t / 1e9, "seconds": t}


def phase_timeline(blk, binding, w, reps, outs, stream, dev, info, R, launches=4):
    """Per-phase block stamps of a few eager launches: for each phase the
    median and max over blocks of (stamp - earliest block start), in us."""
    import torch
    grid = info["cluster_size"] * w.n_kv_heads * (-(-w.batch // info["batch_tile"]))
    bufs = [torch.zeros(grid * binding.TIMELINE_SLOTS, dtype=torch.int64, device=dev)
            for _ in range(launches)]
    per = {n: [] for n in binding.TIMELINE_NAMES}
    gaps = []
    try:
        # back-to-back launches (no host sync in between), one stamp buffer each
        with torch.cuda.stream(stream):
            for i in range(launches):
                r = i % R
                L = reps[r][0]
                binding.cf_set_timeline(blk.handle, bufs[i])
                blk(w.batch, L["hidden"], L["ln_weight"], L["w_qkv"], L["w_o"], L["k_cache"],
                    L["v_cache"], L["positions"], outs[r][0], stream)
        stream.synchronize()
    finally:
        binding.cf_set_timeline(blk.handle, None)
    prev_end = None
    for buf in bufs:
        st = buf.view(grid, binding.TIMELINE_SLOTS)[:, :len(binding.TIMELINE_NAMES)]
        st = st.cpu().double()
        t0 = st[:, 0].min()
        if prev_end is not None:
            gaps.append(float(t0 - prev_end) / 1e3)
        prev_end = st[:, binding.TIMELINE_NAMES.index("end")].max()
        for j, n in enumerate(binding.TIMELINE_NAMES):
            col = st[:, j]
            col = col[col > 0]
            if len(col):
                rel = (col - t0) / 1e3
                per[n].append((float(rel.median()), float(rel.max())))
    res = {n: {"median": round(statistics.median(v[0] for v in vals), 2),
               "max": round(statistics.median(v[1] for v in vals), 2)}
           for n, vals in per.items() if vals}
    if gaps:
        res["gap_to_next_launch"] = {"median": round(statistics.median(gaps), 2),
                                     "max": round(max(gaps), 2)}
    return res


# ---------------------------------------------------------------- oracle --
def time_oracle(w, layer_cpu, budget_s: float, max_steps: int | None = None, wf=None):
    """Run the float64 oracle over batch rows of one step until budget_s is
    spent (at least one row); with an FFN workload ``wf`` each row also runs
    the FFN on the attention block's output (layer_cpu["ffn"] holds its
    tensors).  Returns (seconds per full step, rows done)."""
    import numpy as np
    import oracle
    from attention_block_gb300 import synth

    f = {k: synth.to_f64(layer_cpu[k]) for k in ("hidden", "ln_weight", "w_qkv", "w_o")}
    ff = ({k: synth.to_f64(layer_cpu["ffn"][k]) for k in ("ln_weight", "w_gate", "w_up", "w_down")}
          if wf is not None else None)
    pos = layer_cpu["positions"].numpy()
    cfg = w.oracle_cfg()
    rows_done, t_rows = 0, 0.0
    t0 = time.perf_counter()
    b = 0
    while True:
        kc = np.ascontiguousarray(synth.to_f64(layer_cpu["k_cache"][b]))
        vc = np.ascontiguousarray(synth.to_f64(layer_cpu["v_cache"][b]))
        s = time.perf_counter()
        r = oracle.decode_row(cfg, f["hidden"][b], f["ln_weight"], f["w_qkv"], f["w_o"], kc, vc,
                              int(pos[b]))
        if ff is not None:
            oracle.ffn_row(r["out"], ff["ln_weight"], ff["w_gate"], ff["w_up"], ff["w_down"],
                           wf.rms_eps)
        t_rows += time.perf_counter() - s
        rows_done += 1
        b = (b + 1) % w.batch
        if time.perf_counter() - t0 >= budget_s or (max_steps and rows_done >= max_steps):
            break
    per_row = t_rows / rows_done
    return per_row * w.batch * w.layers, rows_done


# ------------------------------------------------------------------ main --
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cluster-size", type=int, default=int(os.environ.get("CF_CLUSTER_SIZE", 0)))
    ap.add_argument("--batch-tile", type=int, default=int(os.environ.get("CF_BATCH_TILE", 0)))
    ap.add_argument("--stage-bytes", type=int, default=int(os.environ.get("CF_STAGE_BYTES", 0)))
    ap.add_argument("--ctas-per-sm", type=int, default=int(os.environ.get("CF_CTAS_PER_SM", 0)))
    ap.add_argument("--max-stages", type=int, default=int(os.environ.get("CF_MAX_STAGES", 0)))
    ap.add_argument("--ffn", type=int, default=0,
                    help="intermediate size of the gated FFN that follows the attention block "
                         "in every layer (a whole decoder layer per step); 0 = the attention "
                         "block alone")
    ap.add_argument("--rows-per-block", type=int,
                    default=int(os.environ.get("CF_ROWS_PER_BLOCK", 0)))
    ap.add_argument("--pdl", type=int, default=int(os.environ.get("CF_PDL", 0)),
                    help="programmatic dependent launch: 0 default (on), -1 off")
    ap.add_argument("--timeline", action="store_true",
                    help="add per-phase block timings (globaltimer) of a few launches")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--unfused", action="store_true",
                    help="time the three-kernel path with HBM intermediates (the fusion "
                         "baseline) instead of the fused kernel")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ref-budget", type=float, default=0.0,
                    help="--impl reference: seconds of oracle work per step (0 = the run's "
                         "~150 s spread over its steps)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--collectives", action="store_true",
                    help="instead of the decode step: time the DSMEM collectives "
                         "(ClusterReduce all-reduce / reduce-scatter, ClusterGather) for "
                         "cluster sizes 2-16 in SM cycles, one JSON line each")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.collectives:
        return run_collectives(args)

    import torch

    from attention_block_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.workload in synth.MLA_WORKLOADS:
        wm = synth.MLA_WORKLOADS[args.workload]
        if args.impl == "reference":
            return run_mla_reference(args, wm, rank, world)
        return run_mla(args, wm, rank, world, local)
    w = synth.workload(args.workload)

    if args.impl == "reference":
        return run_reference(args, w, rank, world)

    import torch.distributed as dist
    from attention_block_gb300 import binding

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or FALLBACK_L2_BYTES

    # ---- inputs: R replicas (or the 32-layer chain), all resident in HBM
    layer0 = synth.make_layer(w, seed=0, device=dev)
    pos0 = layer0["positions"].tolist()
    step_bytes = algorithmic_bytes(w, pos0) * w.layers
    if w.layers > 1:
        reps = [[layer0] + [synth.make_layer(w, seed=l, device=dev) for l in range(1, w.layers)]]
    else:
        n_rep = max(1, -(-4 * l2 // algorithmic_bytes(w, pos0)))
        reps = [[layer0]] + [[synth.make_layer(w, seed=r, device=dev)] for r in range(1, n_rep)]
    R = len(reps)
    # The whole decoder layer: every layer's attention block is followed by
    # the second RMSNorm + gated FFN + residual, with its own weights.
    wf, ffn_blk = None, None
    if args.ffn > 0:
        wf = synth.custom_ffn(name=f"ffn_i{args.ffn}", hidden=w.hidden, intermediate=args.ffn,
                              batch=w.batch, dtype=w.dtype, rms_eps=w.rms_eps)
        ffn_blk = binding.FfnBlock(w.hidden, args.ffn, w.batch, w.rms_eps, w.dtype)
        for ri, rep in enumerate(reps):
            for li, L in enumerate(rep):
                L["ffn"] = synth.make_ffn(wf, seed=1000 * (ri + 1) + li, device=dev)
                L["h_mid"] = torch.empty_like(L["hidden"])
        step_bytes += ffn_bytes(wf) * w.layers
    footprint = sum(tensor_bytes(L) for rep in reps for L in rep)
    blk = binding.DecodeAttnBlock(
        hidden=w.hidden, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim,
        max_batch=w.batch, s_max=w.s_max, rope_theta=w.rope_theta, rms_eps=w.rms_eps,
        dtype=w.dtype, cluster_size=args.cluster_size, batch_tile=args.batch_tile,
        stage_bytes=args.stage_bytes, ctas_per_sm=args.ctas_per_sm,
        pdl=args.pdl, max_stages=args.max_stages, rows_per_block=args.rows_per_block)
    info = blk.launch_info()
    step_fn = blk.unfused if args.unfused else blk
    kernels_per_layer = 3 if args.unfused else 1
    # the FFN runs one kernel for 1-2 rows, a tensor-core pair for more
    ffn_kernels = ffn_blk.kernels(w.batch)["kernels"] if ffn_blk is not None else 0
    ffn_name = "cf_ffn_kernel" if ffn_kernels <= 1 else "cf_ffn_gu_kernel+cf_ffn_down_kernel"
    outs = [[torch.empty_like(L["hidden"]) for L in rep] for rep in reps]

    stream = torch.cuda.Stream(device=dev)

    def layer_step(x, L, pos, out, ev=None):
        """One layer: the attention block (then the FFN) on `stream`; ev, if
        given, holds events recorded before, between and after."""
        if ev:
            ev[0].record(stream)
        mid = out if ffn_blk is None else L["h_mid"]
        step_fn(w.batch, x, L["ln_weight"], L["w_qkv"], L["w_o"], L["k_cache"], L["v_cache"],
                pos, mid, stream)
        if ev:
            ev[1].record(stream)
        if ffn_blk is not None:
            F = L["ffn"]
            ffn_blk(w.batch, mid, F["ln_weight"], F["w_gate"], F["w_up"], F["w_down"], out, stream)
            if ev:
                ev[2].record(stream)

    def run_step(r):
        x = reps[r][0]["hidden"]
        for l, L in enumerate(reps[r]):
            layer_step(x, L, L["positions"], outs[r][l])
            x = outs[r][l]

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            run_step(i % R)
    stream.synchronize()
    st = blk.status()
    if st != binding.CF_OK:
        raise RuntimeError(f"device status after warm-up: {binding.strerror(st)}")

    # ---- per-launch kernel durations (eager, CUDA events on the launch stream)
    n_lat = min(args.steps, 4 * R if w.layers == 1 else 4)
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3))
           for _ in range(n_lat * w.layers)]
    with torch.cuda.stream(stream):
        k = 0
        for i in range(n_lat):
            r = i % R
            x = reps[r][0]["hidden"]
            for l, L in enumerate(reps[r]):
                layer_step(x, L, L["positions"], outs[r][l], evs[k])
                x = outs[r][l]
                k += 1
    stream.synchronize()
    launch_ms = [e[0].elapsed_time(e[1]) for e in evs]
    launch_ms_avg = sum(launch_ms) / len(launch_ms)
    ffn_ms = [e[1].elapsed_time(e[2]) for e in evs] if ffn_blk is not None else []

    timeline = None
    if args.timeline and ffn_blk is None:
        timeline = phase_timeline(blk, binding, w, reps, outs, stream, dev, info, R)

    # ---- the timed region: graph-captured steps.  One graph holds all R
    # replica steps back to back (so consecutive kernels can overlap their
    # launch through programmatic dependent launch); one-step graphs cover a
    # step count that is not a multiple of R.
    use_graph = not args.no_graph
    single, full = [], None
    if use_graph:
        for r in range(R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                run_step(r)
            single.append(g)
        full = torch.cuda.CUDAGraph()
        with torch.cuda.graph(full, stream=stream):
            for r in range(R):
                run_step(r)
        with torch.cuda.stream(stream):
            for i in range(-(-args.warmup // R)):
                full.replay()
        stream.synchronize()

    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        h0 = time.time()
        with torch.cuda.stream(stream):
            t_start.record(stream)
            if use_graph:
                for _ in range(args.steps // R):
                    full.replay()
                for r in range(args.steps % R):
                    single[r].replay()
            else:
                for i in range(args.steps):
                    run_step(i % R)
            t_end.record(stream)
        stream.synchronize()
        clk.mark(h0, time.time())
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    elapsed_s = t_start.elapsed_time(t_end) / 1e3
    st = blk.status()
    if st != binding.CF_OK:
        raise RuntimeError(f"device status after timed steps: {binding.strerror(st)}")

    # ---- the FFN kernel on its own (its roofline line): graph replays of the
    # FFN launches of every replica and layer, on the attention outputs
    ffn_launch_s = None
    if ffn_blk is not None:
        if ffn_blk.status() != binding.CF_OK:
            raise RuntimeError("FFN device status after timed steps")
        g_ffn = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_ffn, stream=stream):
            for r in range(R):
                for l, L in enumerate(reps[r]):
                    F = L["ffn"]
                    ffn_blk(w.batch, L["h_mid"], F["ln_weight"], F["w_gate"], F["w_up"],
                            F["w_down"], outs[r][l], stream)
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup // R)):
                g_ffn.replay()
        n_ffn = max(1, args.steps // R)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            f0.record(stream)
            for _ in range(n_ffn):
                g_ffn.replay()
            f1.record(stream)
        stream.synchronize()
        ffn_launch_s = f0.elapsed_time(f1) / 1e3 / (n_ffn * R * w.layers)

    # ---- end to end through the public API with host buffers
    B, H = w.batch, w.hidden
    h_in = [torch.empty_like(reps[r][0]["hidden"], device="cpu").pin_memory() for r in range(R)]
    p_in = [torch.empty_like(reps[r][0]["positions"], device="cpu").pin_memory()
            for r in range(R)]
    for r in range(R):
        h_in[r].copy_(reps[r][0]["hidden"])
        p_in[r].copy_(reps[r][0]["positions"])
    h_out = torch.empty_like(h_in[0]).pin_memory()
    x_dev = [torch.empty_like(reps[r][0]["hidden"]) for r in range(R)]
    p_dev = [torch.empty_like(reps[r][0]["positions"]) for r in range(R)]
    e2e_steps = max(args.e2e_steps, 3)

    def e2e_step(i):
        r = i % R
        x_dev[r].copy_(h_in[r], non_blocking=True)
        p_dev[r].copy_(p_in[r], non_blocking=True)
        x = x_dev[r]
        for l, L in enumerate(reps[r]):
            layer_step(x, L, p_dev[r], outs[r][l])
            x = outs[r][l]
        h_out.copy_(outs[r][-1], non_blocking=True)

    # As a serving loop runs it: each step (copy in from pinned memory, the
    # kernel(s), copy the result out) is one graph replay; the copies stay
    # inside the timed region every step.
    e2e_graphs = []
    if use_graph:
        for r in range(R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                e2e_step(r)
            e2e_graphs.append(g)

    def e2e_run(i):
        if e2e_graphs:
            e2e_graphs[i % R].replay()
        else:
            e2e_step(i)

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_run(i)
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(e2e_steps):
            e2e_run(i)
        e1.record(stream)
    stream.synchronize()
    e2e_s = e0.elapsed_time(e1) / 1e3
    h2d = B * H * h_in[0].element_size() + 4 * B
    d2h = B * H * h_out.element_size()

    # ---- whole-job aggregation (max time over ranks)
    mine = [float(step_bytes * args.steps), elapsed_s, float(args.steps)]
    mine_e2e = [float(step_bytes * e2e_steps), e2e_s, float(e2e_steps)]
    rows = allgather_rows(mine + mine_e2e, world, dev)
    per_rank = [r[:3] for r in rows]
    per_rank_e2e = [r[3:] for r in rows]
    agg = aggregate(per_rank)
    agg_e2e = aggregate(per_rank_e2e)

    if rank == 0:
        peak, peak_kind = measured_peak_hbm()
        per_launch_bytes = algorithmic_bytes(w, pos0)
        # The kernel's average launch duration inside the timed region: one
        # kernel per layer, launched back to back on one stream, timed with
        # CUDA events on that stream.
        launch_s_timed = elapsed_s / (args.steps * w.layers)
        kernel_name = ("unfused path: uf_proj_kernel, uf_attn_kernel, uf_proj_kernel"
                       if args.unfused else
                       KERNEL_NAMES.get(info.get("mode", 0), "cf_decode_kernel"))
        traffic = recorded_traffic(w.name)
        layer_kernels = None
        if wf is not None:
            # Two kernels per layer: the attention block's share of the layer
            # time is the layer time less the FFN's (timed alone above); the
            # roofline line is the kernel that takes longer.
            attn_s = max(launch_s_timed - ffn_launch_s, 1e-9)
            layer_kernels = {
                kernel_name: {"us": round(attn_s * 1e6, 3), "bytes": per_launch_bytes,
                              "GBs": round(per_launch_bytes / attn_s / 1e9, 1)},
                ffn_name: {"us": round(ffn_launch_s * 1e6, 3), "bytes": ffn_bytes(wf),
                                  "GBs": round(ffn_bytes(wf) / ffn_launch_s / 1e9, 1),
                                  "timing": "FFN-only graph replays / launches"},
            }
            if ffn_launch_s >= attn_s:
                kernel_name, per_launch_bytes, traffic = ffn_name, ffn_bytes(wf), None
                launch_s_timed = ffn_launch_s
                launch_ms = ffn_ms
                launch_ms_avg = sum(ffn_ms) / len(ffn_ms)
            else:
                launch_s_timed = attn_s
        achieved = per_launch_bytes / launch_s_timed / 1e9
        us_step = elapsed_s / args.steps * 1e6
        cpu = None
        if world == 1:
            lay_cpu = to_cpu(reps[0][0])
            t_cpu, rows = time_oracle(w, lay_cpu, args.cpu_budget, wf=wf)
            cpu = {"value": step_bytes / t_cpu / 1e9, "unit": "GB/s", "cores": 1,
                   "kind": "oracle", "us_per_step": t_cpu * 1e6,
                   "sample": (f"{rows} batch row(s) of layer 0 of this workload through the "
                              f"float64 single-threaded C oracle"
                              f"{' (attention block, then the FFN)' if wf else ''}; "
                              f"per-step time = per-row time "
                              f"x {w.batch} rows x {w.layers} layer(s)"),
                   "host_cpus": os.cpu_count()}
        line = {
            "metric": METRIC,
            "value": round(agg["gbs"], 2),
            "unit": "GB/s",
            "us_per_step": round(us_step, 3),
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(elapsed_s / args.steps * 1e3, 6),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": w.dtype,
            "accumulate": "f32",
            "data": "synthetic",
            "config": {
                "workload": w.name + (f"+ffn_i{args.ffn}" if wf else ""),
                "hidden": w.hidden, "q_heads": w.n_q_heads,
                "kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "batch": w.batch,
                "positions": w.positions, "layers_per_step": w.layers,
                "storage_dtype": w.dtype, "accumulate": "f32",
                "algorithmic_bytes_per_step": step_bytes,
                "flops_per_step": (flops_per_step(w, pos0) + (ffn_flops(wf) if wf else 0))
                * w.layers,
                **({"ffn_intermediate": args.ffn,
                    "ffn_launch": {**ffn_blk.launch_info(), **ffn_blk.kernels(w.batch)}}
                   if wf else {}),
                "l2_defeat": (f"inputs larger than L2: {R} independently seeded replica(s) "
                              f"rotated, {footprint / 1e9:.2f} GB resident vs L2 "
                              f"{l2 / 1e6:.0f} MB"),
                "cuda_graph": use_graph, "parallelism": f"replicas x{world}",
                "launch": info,
                "path": ("unfused (3 kernels, HBM intermediates)" if args.unfused else "fused")
                + (" attention block, then the FFN kernel" if wf else ""),
            },
            "roofline": {
                "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "traffic": traffic,
                "kernel": kernel_name,
                "launch_us_avg": round(launch_s_timed * 1e6, 3),
                "launch_timing": ("timed region (graph replays) / launches" if wf is None else
                                  "dominant kernel of the layer, see layer_kernels"),
                **({"layer_kernels": layer_kernels} if layer_kernels else {}),
                "isolated_launch_us_avg": round(launch_ms_avg * 1e3, 3),
                "isolated_launch_us_min": round(min(launch_ms) * 1e3, 3),
                "bytes_per_launch": per_launch_bytes,
                "frac_of_nominal_7_9TBs": round(achieved / 7900.0, 4),
            },
            "e2e": {"value": round(agg_e2e["gbs"], 2), "unit": "GB/s",
                    "us_per_step": round(e2e_s / e2e_steps * 1e6, 3),
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "cuda_graph": bool(e2e_graphs)},
            "gpu_launches": args.steps * w.layers * (kernels_per_layer + ffn_kernels),
            **({"timeline_us": timeline} if timeline else {}),
            "clocks": clk.result(),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    blk.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------- MLA variant --
MLA_TENSORS = ("hidden", "ln_weight", "w_q", "w_dkv", "kv_norm_weight", "w_ukv", "w_o")


def mla_bytes(w, positions) -> int:
    """Bytes one MLA decode step must move at minimum: every weight once, the
    latent cache rows [0, p_b) of every row, the new latent row written,
    hidden read, out written, positions."""
    es = 4 if w.dtype == "f32" else 2
    nh, dn, dr, dv, dc, H = w.n_heads, w.d_nope, w.d_rope, w.d_v, w.d_latent, w.hidden
    weights = (H * nh * (dn + dr) + H * (dc + dr) + dc * nh * (dn + dv) + nh * dv * H + H
               + dc) * es
    cache = sum(int(p) * (dc + dr) * es for p in positions) + w.batch * (dc + dr) * es
    return weights + cache + 2 * w.batch * H * es + 4 * w.batch


def run_mla(args, w, rank, world, local):
    """The MLA variant's decode step (cf_mla_decode), timed like the attention
    block: graph replays over replicas spanning >= 4x L2, CUDA events on the
    launching stream, max over ranks; e2e with host buffers; the float64
    oracle as the CPU baseline."""
    import torch
    import torch.distributed as dist

    from attention_block_gb300 import binding, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or FALLBACK_L2_BYTES
    layer0 = synth.make_mla_layer(w, seed=0, device=dev)
    pos0 = layer0["positions"].tolist()
    step_bytes = mla_bytes(w, pos0)
    n_rep = max(1, -(-4 * l2 // step_bytes))
    reps = [layer0] + [synth.make_mla_layer(w, seed=r, device=dev) for r in range(1, n_rep)]
    R = len(reps)
    footprint = sum(tensor_bytes(L) for L in reps)
    blk = binding.MlaBlock(w.hidden, w.n_heads, w.batch, w.s_max, w.rope_theta, w.rms_eps,
                           w.dtype, w.d_nope, w.d_rope, w.d_v, w.d_latent)
    info = blk.launch_info()
    outs = [torch.empty_like(L["hidden"]) for L in reps]
    stream = torch.cuda.Stream(device=dev)

    def step(r, x=None, pos=None, ev=None):
        L = reps[r]
        args_ = [L[k] for k in MLA_TENSORS]
        if x is not None:
            args_[0] = x
        if ev:
            ev[0].record(stream)
        blk(w.batch, *args_, L["latent_cache"], L["positions"] if pos is None else pos, outs[r],
            stream)
        if ev:
            ev[1].record(stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i % R)
    stream.synchronize()
    if blk.status() != binding.CF_OK:
        raise RuntimeError("MLA device status after warm-up")
    n_lat = min(args.steps, 4 * R)
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(n_lat)]
    with torch.cuda.stream(stream):
        for i in range(n_lat):
            step(i % R, ev=evs[i])
    stream.synchronize()
    launch_ms = [e[0].elapsed_time(e[1]) for e in evs]
    use_graph = not args.no_graph
    single, full = [], None
    if use_graph:
        for r in range(R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(r)
            single.append(g)
        full = torch.cuda.CUDAGraph()
        with torch.cuda.graph(full, stream=stream):
            for r in range(R):
                step(r)
        with torch.cuda.stream(stream):
            for _ in range(-(-args.warmup // R)):
                full.replay()
        stream.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        h0 = time.time()
        with torch.cuda.stream(stream):
            t_start.record(stream)
            if use_graph:
                for _ in range(args.steps // R):
                    full.replay()
                for r in range(args.steps % R):
                    single[r].replay()
            else:
                for i in range(args.steps):
                    step(i % R)
            t_end.record(stream)
        stream.synchronize()
        clk.mark(h0, time.time())
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    elapsed_s = t_start.elapsed_time(t_end) / 1e3
    if blk.status() != binding.CF_OK:
        raise RuntimeError("MLA device status after timed steps")
    # end to end: hidden rows and positions from pinned host memory, out back
    h_in = [L["hidden"].cpu().pin_memory() for L in reps]
    p_in = [L["positions"].cpu().pin_memory() for L in reps]
    h_out = torch.empty_like(h_in[0]).pin_memory()
    x_dev = [torch.empty_like(L["hidden"]) for L in reps]
    p_dev = [torch.empty_like(L["positions"]) for L in reps]

    def e2e_step(i):
        r = i % R
        x_dev[r].copy_(h_in[r], non_blocking=True)
        p_dev[r].copy_(p_in[r], non_blocking=True)
        step(r, x=x_dev[r], pos=p_dev[r])
        h_out.copy_(outs[r], non_blocking=True)

    e2e_steps = max(args.e2e_steps, 3)
    e2e_graphs = []
    if use_graph:
        for r in range(R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                e2e_step(r)
            e2e_graphs.append(g)
    run = (lambda i: e2e_graphs[i % R].replay()) if e2e_graphs else e2e_step
    with torch.cuda.stream(stream):
        for i in range(3):
            run(i)
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(e2e_steps):
            run(i)
        e1.record(stream)
    stream.synchronize()
    e2e_s = e0.elapsed_time(e1) / 1e3
    rows = allgather_rows([float(step_bytes * args.steps), elapsed_s, float(args.steps),
                           float(step_bytes * e2e_steps), e2e_s, float(e2e_steps)], world, dev)
    agg = aggregate([r[:3] for r in rows])
    agg_e2e = aggregate([r[3:] for r in rows])
    if rank == 0:
        peak, peak_kind = measured_peak_hbm()
        launch_s = elapsed_s / args.steps
        achieved = step_bytes / launch_s / 1e9
        cpu = None
        if world == 1:
            cpu = time_mla_oracle(w, reps[0], args.cpu_budget)
        B, H = w.batch, w.hidden
        line = {
            "metric": METRIC, "value": round(agg["gbs"], 2), "unit": "GB/s",
            "us_per_step": round(elapsed_s / args.steps * 1e6, 3), "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed_s / args.steps * 1e3, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "accumulate": "f32",
            "data": "synthetic",
            "config": {"workload": w.name, "variant": "DeepSeek MLA (latent KV cache)",
                       "hidden": H, "heads": w.n_heads, "d_nope": w.d_nope, "d_rope": w.d_rope,
                       "d_v": w.d_v, "d_latent": w.d_latent, "batch": B,
                       "positions": w.positions, "storage_dtype": w.dtype,
                       "algorithmic_bytes_per_step": step_bytes,
                       "l2_defeat": (f"inputs larger than L2: {R} independently seeded "
                                     f"replica(s) rotated, {footprint / 1e9:.2f} GB resident vs "
                                     f"L2 {l2 / 1e6:.0f} MB"),
                       "cuda_graph": use_graph, "parallelism": f"replicas x{world}",
                       "launch": info},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_kind == "measured" else "fallback 6.8 TB/s",
                         "traffic": recorded_traffic(w.name, MLA_KERNEL_ROOTS),
                         "kernel": "cf_mla_kernel",
                         "launch_us_avg": round(launch_s * 1e6, 3),
                         "launch_timing": "timed region (graph replays) / launches",
                         "isolated_launch_us_avg": round(sum(launch_ms) / len(launch_ms) * 1e3, 3),
                         "bytes_per_launch": step_bytes,
                         "frac_of_nominal_7_9TBs": round(achieved / 7900.0, 4)},
            "e2e": {"value": round(agg_e2e["gbs"], 2), "unit": "GB/s",
                    "us_per_step": round(e2e_s / e2e_steps * 1e6, 3),
                    "h2d_bytes_per_step": B * H * h_in[0].element_size() + 4 * B,
                    "d2h_bytes_per_step": B * H * h_out.element_size(),
                    "steps": e2e_steps, "cuda_graph": bool(e2e_graphs)},
            "gpu_launches": args.steps,
            "clocks": clk.result(),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    blk.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def time_mla_oracle(w, layer, budget_s: float):
    """The float64 MLA oracle on one host core over batch rows of one step
    until budget_s is spent (at least one row), scaled to a full step."""
    import oracle
    from attention_block_gb300 import synth

    f = {k: synth.to_f64(layer[k]) for k in MLA_TENSORS}
    pos = layer["positions"].tolist()
    rows, t_rows, b = 0, 0.0, 0
    t0 = time.perf_counter()
    while True:
        lc = synth.to_f64(layer["latent_cache"][b]).copy()
        s = time.perf_counter()
        oracle.mla_row(w.oracle_cfg(), f["hidden"][b], f["ln_weight"], f["w_q"], f["w_dkv"],
                       f["kv_norm_weight"], f["w_ukv"], f["w_o"], lc, int(pos[b]))
        t_rows += time.perf_counter() - s
        rows += 1
        b = (b + 1) % w.batch
        if time.perf_counter() - t0 >= budget_s:
            break
    t_step = t_rows / rows * w.batch
    return {"value": mla_bytes(w, pos) / t_step / 1e9, "unit": "GB/s", "cores": 1,
            "kind": "oracle", "us_per_step": t_step * 1e6,
            "sample": (f"{rows} batch row(s) of one layer through the float64 single-threaded "
                       f"C MLA oracle; per-step time = per-row time x {w.batch} rows"),
            "host_cpus": os.cpu_count()}


def run_mla_reference(args, w, rank, world):
    """The float64 MLA oracle as the reference arm, host cores, rank 0 only."""
    if rank != 0:
        return 0
    from attention_block_gb300 import synth

    layer = synth.make_mla_layer(w, seed=0, device="cpu")
    budget = (args.ref_budget if args.ref_budget > 0
              else max(1.0, 150.0 / max(1, args.steps + args.warmup)))
    times = [time_mla_oracle(w, layer, budget)["us_per_step"] for _ in range(args.steps)]
    t = sum(times) / len(times) / 1e6
    step_bytes = mla_bytes(w, layer["positions"].tolist())
    val = step_bytes / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s",
            "us_per_step": round(t * 1e6, 1), "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "variant": "DeepSeek MLA (latent KV cache)",
                       "batch": w.batch, "positions": w.positions,
                       "algorithmic_bytes_per_step": step_bytes},
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": 1,
                             "kind": "oracle",
                             "sample": f"each step: rows of one layer through the float64 MLA "
                                       f"oracle for ~{budget:.1f} s, scaled to {w.batch} rows",
                             "host_cpus": os.cpu_count()},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# The collectives timed by --collectives: (name, kind of cf_bench_cluster_collective,
# floats per block for a given total payload and cluster size).  The totals
# follow the 128 KB payload of the pages' primitive latency table: for the
# all-reduce the blocks' contributions sum to it, for the gather it is what
# every block ends up holding, for the reduce-scatter it is each block's input
# (64 KB: the receive buffers must fit next to it in shared memory).
COLLECTIVES = (
    ("allreduce_sum", 0, lambda total, N: total // (4 * N)),
    ("allreduce_max", 1, lambda total, N: total // (4 * N)),
    ("reduce_scatter", 2, lambda total, N: total // 2 // (4 * N)),
    ("gather", 3, lambda total, N: total // (4 * N)),
)


def run_collectives(args):
    """Median over repeats of the slowest block's SM cycles inside one
    collective, and that time in microseconds at the sampled SM clock."""
    import torch

    from attention_block_gb300 import binding

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    total = 128 * 1024
    reps = max(5, min(args.steps, 50))
    with ClockSampler(dev.index) as clk:
        rows = []
        for name, kind, per_block in COLLECTIVES:
            for N in (2, 4, 8, 16):
                n = per_block(total, N)
                length = N * n if kind >= 2 else n
                x = torch.randn(N, length, device=dev)
                out = torch.empty(N, N * n if kind == 3 else (n if kind == 2 else length),
                                  device=dev)
                err = torch.zeros(1, dtype=torch.int32, device=dev)
                cyc = torch.zeros(N, dtype=torch.int64, device=dev)
                got = []
                for i in range(args.warmup + reps):
                    rc = binding.cf_bench_cluster_collective(kind, N, n, x, out, err, cyc)
                    if rc != binding.CF_OK:
                        raise RuntimeError(f"{name} N={N}: {binding.strerror(rc)}")
                    torch.cuda.synchronize()
                    if i >= args.warmup:
                        got.append(int(cyc.max().item()))
                if int(err.item()) != 0:
                    raise RuntimeError(f"{name} N={N}: device error {int(err.item())}")
                rows.append((name, N, n, statistics.median(got)))
    clocks = clk.result()
    mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or 2070.0
    for name, N, n, cyc in rows:
        payload = (N * n if name != "reduce_scatter" else N * n) * 4
        print(json.dumps({"collective": name, "cluster_size": N, "floats_per_block": n,
                          "payload_bytes": payload, "cycles": cyc,
                          "us": round(cyc / mhz, 3), "sm_mhz": mhz,
                          "rounds": (N - 1).bit_length(), "clocks": clocks}), flush=True)
    return 0


def run_reference(args, w, rank, world):
    """The float64 oracle as the reference arm, on the host cores, rank 0 only."""
    if rank != 0:
        return 0
    import torch

    from attention_block_gb300 import synth

    layer = synth.make_layer(w, seed=0, device="cpu")
    pos = layer["positions"].tolist()
    step_bytes = algorithmic_bytes(w, pos) * w.layers
    wf = None
    if args.ffn > 0:
        wf = synth.custom_ffn(name=f"ffn_i{args.ffn}", hidden=w.hidden, intermediate=args.ffn,
                              batch=w.batch, dtype=w.dtype, rms_eps=w.rms_eps)
        layer["ffn"] = synth.make_ffn(wf, seed=1000, device="cpu")
        step_bytes += ffn_bytes(wf) * w.layers
    budget = (args.ref_budget if args.ref_budget > 0
              else max(1.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        time_oracle(w, layer, 0.0, max_steps=1, wf=wf)
    times, rows_total = [], 0
    for _ in range(args.steps):
        t_step, rows = time_oracle(w, layer, budget, wf=wf)
        times.append(t_step)
        rows_total += rows
    t = sum(times) / len(times)
    val = step_bytes / t / 1e9
    sample = (f"each step: batch rows of layer 0 through the float64 single-threaded C oracle "
              f"for ~{budget:.1f} s; per-step time = per-row time x {w.batch} rows x "
              f"{w.layers} layer(s); {rows_total} rows in total")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s",
        "us_per_step": round(t * 1e6, 1), "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name + (f"+ffn_i{args.ffn}" if wf else ""),
                   "hidden": w.hidden, "q_heads": w.n_q_heads,
                   "kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "batch": w.batch,
                   "positions": w.positions, "layers_per_step": w.layers,
                   "storage_dtype": w.dtype, "algorithmic_bytes_per_step": step_bytes,
                   **({"ffn_intermediate": args.ffn} if wf else {})},
        "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample, "host_cpus": os.cpu_count()},
        "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
