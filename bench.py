"""Throughput of the CSA decode hot path (compress -> lightning indexer top-k -> attention -> window
commit) on the 32-sequence x 131072-token workload: 64 query heads, shared KV dim 512 (448 FP8 +
64 BF16 RoPE dims), m=4 overlapped compression (32768 entries per sequence), indexer rank 128 with
4 heads in FP4 E2M1 with per-32 UE8M0 scales, top-k 512, window 128.

One step = one decode token for every sequence through the whole path.  Inputs are seeded
synthetic tensors already resident in HBM; L2 is flushed (a 256 MB write) between timed steps.
Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

WL = synth.CONFIGS["csa_decode"]
METRIC = "CSA/HCA attention queries/s at 128K-1M ctx"
# DRAM bytes (read + write) per step of the attention and of the indexer on the csa_decode
# workload, from one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum), together with
# the hash of the kernel sources they were taken on: when the sources differ from that hash the
# counters no longer describe the kernels that run and `traffic` is reported as null.
TRAFFIC = {"source_sha1": "ed92e68e5bf6e37899e63376ba67e52d88c4cbef",
           "attend": 29762901,    # attend_tc1_kernel (top-k part 14.50 MB + window part 4.68 MB) + combine 10.58 MB
           "index": 71652181}     # index_tc_kernel<4, 4, 1, 6>: 71.60 MB read + 0.05 MB written (mean of 3 launches)
UNIT = "queries/s"


# measured after the headline by default: the other configurations and the tensor-pipe probe
OTHER_WORKLOADS = ("csa_decode_1m", "hca_decode", "mixed_decode", "csa_prefill", "compress_1m", "tensor_peak")


def run_others(args):
    """The other workloads, each as `bench.py --workload W` in a child process on this GPU (no
    torchrun variables: a plain one-GPU run), their JSON lines condensed for the headline line."""
    import subprocess
    names = OTHER_WORKLOADS if args.others == "auto" else tuple(w for w in args.others.split(",") if w)
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "LOCAL_WORLD_SIZE", "MASTER_ADDR", "MASTER_PORT",
                        "GROUP_RANK", "ROLE_RANK", "TORCHELASTIC_RUN_ID")}
    out = {}
    for w in names:
        cmd = [sys.executable, os.path.abspath(__file__), "--workload", w, "--steps", str(min(args.steps, 10)),
               "--warmup", str(max(3, min(args.warmup, 5))), "--no-cpu-baseline", "--others", "none"]
        try:
            r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
            lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
            if r.returncode != 0 or not lines:
                out[w] = {"error": f"exit {r.returncode}: {(r.stderr or '').strip().splitlines()[-1:]}"}
                continue
            d = json.loads(lines[-1])
            keep = {k: d.get(k) for k in ("metric", "value", "unit", "ms_per_step", "steps", "warmup", "dtype",
                                          "gpu_launches", "device_status_ok")}
            keep["workload"] = (d.get("config") or {}).get("workload")
            rf = d.get("roofline") or {}
            keep["roofline"] = {k: rf.get(k) for k in ("kernel", "bound", "achieved", "peak", "unit", "frac")}
            if d.get("roofline_step"):
                rs = d["roofline_step"]
                keep["roofline_step"] = {k: rs.get(k) for k in ("achieved", "peak", "unit", "frac")}
            if d.get("rates"):
                keep["rates"] = d["rates"]
            ck = d.get("clocks") or {}
            keep["clocks"] = {k: ck.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")}
            out[w] = keep
        except Exception as e:   # a failed extra line never costs the headline
            out[w] = {"error": repr(e)[:200]}
    return out


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="csa_decode",
                    choices=["csa_decode", "csa_decode_1m", "hca_decode", "mixed_decode", "csa_prefill",
                             "compress_1m", "index_key_quantize", "attention_sink", "attend_separate_v", "tensor_peak"],
                    help="csa_decode is the headline line; the others measure the 1M-context CSA decode, the "
                         "HCA decode, the mixed ragged multi-layer and the CSA prefill workloads, and the "
                         "compression of a 1M-token context, with the same timing rules")
    ap.add_argument("--ctx-len", type=int, default=None,
                    help="csa_prefill only: cached tokens instead of the workload's 1,048,576 (a smaller case of "
                         "the same kernels, for profiler captures; the line then names the changed workload)")
    ap.add_argument("--new-tokens", type=int, default=None,
                    help="csa_prefill only: new tokens (queries) instead of the workload's 16,384")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="csa_decode / csa_decode_1m only: sequences instead of the workload's 32 (a smaller case "
                         "of the same kernels, for profiler captures; the line then names the changed workload and "
                         "measures no other workloads)")
    ap.add_argument("--others", default="auto",
                    help="comma-separated workloads measured after the headline (csa_decode, one GPU only), each "
                         "in a process of its own, and summarised in the headline line under 'other_workloads'; "
                         "'auto': " + ",".join(OTHER_WORKLOADS) + "; 'none': the headline alone")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ---- multi-rank logic: every rank serves its own sequences (weak scaling, no data-path
#      collective); the ranks meet only at a barrier before the timed steps and to take the
#      slowest rank's step time

def rank_seed(seed: int, rank: int) -> int:
    """Seed of a rank's own sequences (independent problems per rank)."""
    return seed + 1000 * rank


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's step time (every rank gets it)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(per_rank_units: float, world: int, ms: float) -> float:
    """Whole-job throughput: the units all ranks processed per step over the slowest step time."""
    return per_rank_units * world / (ms * 1e-3)


def workload_config(extra=None, wl=None):
    wl = wl or WL
    cfg = {"workload": wl.name, "num_seqs": wl.num_seqs, "ctx_len": wl.ctx_len, "new_tokens_per_seq": 1,
           "heads": wl.heads, "kv_dim": wl.dim, "row_format": "fp8_e4m3(448)+bf16_rope(64)+f32_scale",
           "m": wl.m, "overlap": True, "index_heads": wl.index_heads, "index_rank": wl.index_rank,
           "index_format": "fp4_e2m1+ue8m0/32", "top_k": wl.top_k, "window": wl.window, "seed": wl.seed,
           "l2": "flushed between timed steps (256 MB write)", "data": "synthetic"}
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"lcsa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1])); mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def kernel_source_sha1() -> str:
    """sha1 over the library's kernel sources (file names and contents, sorted by name)."""
    import hashlib
    h = hashlib.sha1()
    d = os.path.join(ROOT, "long_context_sparse_24_b300", "csrc")
    for name in sorted(os.listdir(d)):
        if name.endswith((".cu", ".cuh")):
            h.update(name.encode())
            with open(os.path.join(d, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def traffic_of(part: str, workload: str):
    """ncu DRAM bytes of `part` if they were captured on the kernel sources that run and on this
    workload (the table holds the csa_decode step's), else None."""
    if workload == WL.name and TRAFFIC.get("source_sha1") and TRAFFIC["source_sha1"] == kernel_source_sha1():
        return TRAFFIC.get(part)
    return None


def graph_kernel_count(graph):
    """Kernel nodes of a captured CUDA graph (the step's launches of this library's kernels), read
    back through the CUDA runtime; None when the graph cannot be inspected."""
    try:
        from cuda.bindings import runtime as cr
        g = cr.cudaGraph_t(init_value=int(graph.raw_cuda_graph()))
        err, _, n = cr.cudaGraphGetNodes(g, 0)
        if err != cr.cudaError_t.cudaSuccess:
            return None
        err, nodes, n = cr.cudaGraphGetNodes(g, n)
        if err != cr.cudaError_t.cudaSuccess:
            return None
        kinds = [cr.cudaGraphNodeGetType(nd) for nd in nodes[:n]]
        return sum(1 for e, t in kinds if e == cr.cudaError_t.cudaSuccess and
                   t == cr.cudaGraphNodeType.cudaGraphNodeTypeKernel)
    except Exception:
        return None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6400.0), "measured"
    return 6400.0, "fallback"


# ---------------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------------

def run_gpu(args, rank, world, local, wl=None):
    wl = wl or WL
    import torch
    import synth.gpu as sg
    import long_context_sparse_24_b300 as lcsa
    from long_context_sparse_24_b300.layer import Layer

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if lcsa.lcs_device_check() != 0:
        raise SystemExit("liblcsa needs a compute-capability 10.3 GPU")
    S, L, H, D = wl.num_seqs, wl.ctx_len, wl.heads, wl.dim
    Hi, r, k, m = wl.index_heads, wl.index_rank, wl.top_k, wl.m
    n_stage = 5                              # extra replays of an instrumented graph (stage times)
    steps_total = args.warmup + args.steps + n_stage
    cap = L + 128 * math.ceil((steps_total + 1) / 128) + 256
    seed = rank_seed(wl.seed, rank)         # each rank serves its own sequences
    layer = Layer("csa", S, cap, H, D, lcsa.LCS_ROW_FP8_SPLIT, m, top_k=k, index_heads=Hi, index_rank=r,
                  max_new=1, device=dev)
    # compressor parameters (w ~ N(0,1)/16, bias ~ N(0,1)/2)
    w = synth.bf16_bits_to_f32(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_W), 0, D)) / 16
    bias = synth.bf16_bits_to_f32(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_B), 0, 2 * m)) / 2
    layer.set_compressor(torch.from_numpy(w.astype(np.float32)).to(dev),
                         torch.from_numpy(bias.astype(np.float32)).to(dev))
    # ---- build the cached context: L raw tokens per sequence, compressed by the library
    chunk = 16384
    raw_chunk = torch.empty((S * chunk, D), dtype=torch.bfloat16, device=dev)
    for c0 in range(0, L, chunk):
        n = min(chunk, L - c0)
        for b in range(S):
            sg.normal_bf16(raw_chunk[b * n:(b + 1) * n], seed, synth.tensor_id(synth.RAW, 0, b), c0 * D)
        layer.fill(layer.batch([c0 + n] * S, [n] * S), raw_chunk[:S * n])
    del raw_chunk
    # ---- indexer keys of every entry the run will create (identity paging: contiguous per sequence)
    bps = layer.cache.paging.max_blocks_per_seq
    n_ent = cap // m
    for b in range(S):
        r0 = b * bps * 32
        sg.e2m1_packed(layer.cache.keys.fp4[r0:r0 + n_ent], seed, synth.tensor_id(synth.IDX_K, 0, b), 0)
        sg.ue8m0(layer.cache.keys.scale[r0:r0 + n_ent], seed, synth.tensor_id(synth.IDX_KS, 0, b), 0)
    # ---- per-step inputs (decode token L+s of every sequence)
    raw_steps = torch.empty((steps_total, S, D), dtype=torch.bfloat16, device=dev)
    q_steps = torch.empty((steps_total, S, H, D), dtype=torch.bfloat16, device=dev)
    iq_steps = torch.empty((steps_total, S, Hi, r // 2), dtype=torch.uint8, device=dev)
    iqs_steps = torch.empty((steps_total, S, Hi, r // 32), dtype=torch.uint8, device=dev)
    hw_np = np.stack([synth.head_weights(seed, synth.tensor_id(synth.HEAD_W, 0, b), L * Hi, steps_total * Hi)
                      .reshape(steps_total, Hi) for b in range(S)], axis=1)
    hw_steps = torch.from_numpy(np.ascontiguousarray(hw_np)).to(dev)
    for s in range(steps_total):
        t = L + s
        for b in range(S):
            sg.normal_bf16(raw_steps[s, b], seed, synth.tensor_id(synth.RAW, 0, b), t * D)
            sg.normal_bf16(q_steps[s, b], seed, synth.tensor_id(synth.QUERY, 0, b), t * H * D)
            sg.e2m1_packed(iq_steps[s, b], seed, synth.tensor_id(synth.IDX_Q, 0, b), t * Hi * r)
            sg.ue8m0(iqs_steps[s, b], seed, synth.tensor_id(synth.IDX_QS, 0, b), t * Hi * r // 32)
    # ---- static step buffers + CUDA graph of one step
    raw_in = torch.empty((S, D), dtype=torch.bfloat16, device=dev)
    q_in = torch.empty((S, H, D), dtype=torch.bfloat16, device=dev)
    iq_in = torch.empty((S, Hi, r // 2), dtype=torch.uint8, device=dev)
    iqs_in = torch.empty((S, Hi, r // 32), dtype=torch.uint8, device=dev)
    hw_in = torch.empty((S, Hi), dtype=torch.float32, device=dev)
    out = torch.empty((S, H, D), dtype=torch.bfloat16, device=dev)
    cu_new = torch.arange(S + 1, dtype=torch.int32, device=dev)
    seq_len = torch.full((S,), L + 1, dtype=torch.int32, device=dev)
    batch = layer.batch([cap] * S, [1] * S, cu_new=cu_new, seq_len=seq_len)

    def load_step(s):
        raw_in.copy_(raw_steps[s]); q_in.copy_(q_steps[s]); iq_in.copy_(iq_steps[s])
        iqs_in.copy_(iqs_steps[s]); hw_in.copy_(hw_steps[s]); seq_len.fill_(L + s + 1)

    STAGES = ["compress", "attend_window", "index_topk", "attend_topk", "window_commit"]
    try:
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(STAGES) + 1)]
    except TypeError:  # torch without event-record nodes in graphs: no stage breakdown
        evs = None
    from long_context_sparse_24_b300 import csa_attend_topk, csa_attend_window

    def step_body(with_events=True):
        if not with_events:
            # the timed step: compression and the window part of attention (side stream) next to
            # the indexer, which leaves them SMs; then the top-k part of attention with the merge
            layer.step(batch, raw_in, q_in, out, idx_q_fp4=iq_in, idx_q_scale=iqs_in, head_w=hw_in)
            return
        # the same calls, serialised on one stream with an event node after each
        c = layer.cache
        calls = [lambda: layer.compress(batch, raw_in),
                 lambda: csa_attend_window(batch, q_in, H, k, m, c.entries, c.paging, c.state, layer.scale,
                                           layer.attend_ws, layer.attend_ws_bytes, layer.status),
                 lambda: layer.select(batch, iq_in, iqs_in, hw_in, spare_sms=layer.window_ctas(batch)),
                 lambda: csa_attend_topk(batch, q_in, H, layer.topk_idx, layer.topk_cnt, k, m, c.entries, c.paging,
                                         c.state, layer.scale, out, None, layer.attend_ws, layer.attend_ws_bytes,
                                         layer.status),
                 lambda: layer.commit(batch)]
        if evs:
            evs[0].record()
        for i, fn in enumerate(calls):
            fn()
            if evs:
                evs[i + 1].record()

    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    # warm-up step 0 runs eagerly (first launches set the kernels' shared-memory attributes);
    # the step is then captured once and replayed for every later decode position
    load_step(0)
    step_body(with_events=False)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph(keep_graph=True)   # the timed step: kernels only
    with torch.cuda.graph(graph):
        step_body(with_events=False)
    graph.instantiate()
    graph_kernels = graph_kernel_count(graph)
    graph_ev = torch.cuda.CUDAGraph()          # the same step with event nodes between the calls
    with torch.cuda.graph(graph_ev):
        step_body(with_events=True)
    timed_end = args.warmup + args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps_total)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps_total)]
    stage_ms = []
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for s in range(1, timed_end):
            load_step(s)
            flush.zero_()
            starts[s].record()
            graph.replay()
            ends[s].record()
        torch.cuda.synchronize()
    for s in range(timed_end, steps_total):      # stage breakdown (not part of the timed steps)
        load_step(s)
        flush.zero_()
        graph_ev.replay()
        torch.cuda.synchronize()
        if evs:
            stage_ms.append([evs[i].elapsed_time(evs[i + 1]) for i in range(len(STAGES))])
    status_ok = True
    if int(layer.status.item()) != 0:
        status_ok = False
    per_step = [starts[s].elapsed_time(ends[s]) for s in range(args.warmup, timed_end)]
    ms = statistics.mean(per_step)
    ms = max_over_ranks(ms, world, dev)
    stages = ([statistics.mean(x[i] for x in stage_ms) for i in range(len(STAGES))] if stage_ms
              else [float("nan")] * len(STAGES))
    stage = dict(zip(STAGES, stages))
    splits_used = layer.attend_ws_bytes > 0
    # compress (entries + state) + indexer (score + select) + attention (tensor-core plan: window part,
    # top-k part, merge; otherwise one kernel, plus a merge when split) + window commit
    tc_plan = D == 512 and H <= 64 and k <= 2048
    attend_launches = 3 if tc_plan else (2 if splits_used else 1)
    launches_per_step = 2 + 1 + attend_launches + (0 if layer.ring_only else 1)
    if graph_kernels is not None:   # counted from the captured step itself
        launches_per_step = graph_kernels
    hbm, peak_kind = measured_peaks()
    peak_src = f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback"
    n_vis = [(L + s + 1) // m for s in range(timed_end, steps_total)]
    # ---- algorithmic bytes per step.  Attention: (k + window) rows of 580 B per query, the query and
    #      the output (H x D BF16 each); 4*H*D FLOP per row (about 167 FLOP/B, below the F16 tensor
    #      balance point of ~270 FLOP/B on this part, so HBM is the roof).  Indexer: 68 B of key per
    #      visible entry per query, the query codes, scales and head weights, and the selection.
    att_bytes = S * ((k + 128) * (D - 64 + 128 + 4) + 2 * H * D * 2)
    att_ms = stage["attend_window"] + stage["attend_topk"]
    key_bytes = r // 2 + r // 32
    idx_bytes = statistics.mean(S * (n * key_bytes + Hi * key_bytes + Hi * 4 + k * 4 + 4) for n in n_vis)
    idx_ms = stage["index_topk"]
    comp_bytes = S * (D * 2 + (D - 64 + 128 + 4))     # one raw row in, one window row out per sequence
    step_bytes = att_bytes + idx_bytes + comp_bytes

    def roof(kernel, nbytes, t_ms, traffic, timing):
        ach = nbytes / (t_ms * 1e-3) / 1e9
        return {"kernel": kernel, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 4), "peak_source": peak_src, "algorithmic_bytes_per_launch": int(nbytes),
                "traffic": traffic, "timing": timing}

    timing = "CUDA events around the call(s) in a serialised copy of the step (event nodes in a CUDA graph)"
    roofline_att = roof("csa_attend_window + csa_attend_topk (attention kernels incl. the merge)", att_bytes,
                        att_ms, traffic_of("attend", wl.name), timing)
    roofline_att["flop_per_step"] = int(S * 4 * H * D * (k + 128))
    roofline_idx = roof("csa_index_topk (scorer and selection)", idx_bytes, idx_ms, traffic_of("index", wl.name),
                        timing)
    roofline_step = roof("whole step (compression, indexer, attention)", step_bytes, ms, None,
                         "CUDA events around each timed step (the graph as it runs)")
    # the dominant stage by device time is the line's roofline; the other stage and the whole step beside it
    if att_ms >= idx_ms:
        roofline, roofline_other = roofline_att, roofline_idx
    else:
        roofline, roofline_other = roofline_idx, roofline_att
    # ---- end to end through the public API with host buffers (pinned), copies in the timed region
    e2e = run_e2e(torch, layer, batch, graph, raw_in, q_in, iq_in, iqs_in, hw_in, out, seq_len, raw_steps,
                  q_steps, iq_steps, iqs_steps, hw_steps, args, L, S, flush)
    return {"ms": ms, "stages": stage, "clocks": clk.summary(), "roofline": roofline,
            "roofline_other": roofline_other, "roofline_step": roofline_step, "e2e": e2e,
            "launches": launches_per_step * args.steps, "status_ok": status_ok,
            "per_rank_queries": S}


# ---------------------------------------------------------------------------------------------
# GPU arm, other workloads: HCA decode (one HCA layer) and the mixed ragged stack (CSA/HCA x 4)
# ---------------------------------------------------------------------------------------------

def run_gpu_stack(args, rank, world, local, wl):
    import torch
    import synth.gpu as sg
    import long_context_sparse_24_b300 as lcsa
    from long_context_sparse_24_b300.model import HybridStack

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if lcsa.lcs_device_check() != 0:
        raise SystemExit("liblcsa needs a compute-capability 10.3 GPU")
    S, H, D = wl.num_seqs, wl.heads, wl.dim
    Hi, r, k = wl.index_heads, wl.index_rank, wl.top_k
    seed = rank_seed(wl.seed, rank)
    if wl.kind == "mixed":
        lengths = [int(x) for x in synth.mixed_lengths(seed, S)]
        n_layers, first = wl.layers, "csa"
    else:
        lengths = [wl.ctx_len] * S
        n_layers, first = 1, "hca"
    steps_total = args.warmup + args.steps
    cap = max(lengths) + 128 * math.ceil((steps_total + 1) / 128) + 256
    stack = HybridStack(n_layers, S, cap, H, D, lcsa.LCS_ROW_FP8_SPLIT, csa_m=4, hca_m=128, top_k=k,
                        index_heads=Hi, index_rank=r, max_new=1, first=first, device=dev)
    # ---- per layer: compressor parameters, the cached context (ragged), indexer keys
    chunk = 16384 if S <= 32 else 8192
    raw_chunk = torch.empty((S * chunk, D), dtype=torch.bfloat16, device=dev)
    for li, layer in enumerate(stack.layers):
        m = layer.m
        nb = 2 * m if layer.overlap else m
        w = synth.bf16_bits_to_f32(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_W, li), 0, D)) / 16
        bias = synth.bf16_bits_to_f32(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_B, li), 0, nb)) / 2
        layer.set_compressor(torch.from_numpy(w.astype(np.float32)).to(dev),
                             torch.from_numpy(bias.astype(np.float32)).to(dev))
        for c0 in range(0, max(lengths), chunk):
            ns = [max(0, min(chunk, L - c0)) for L in lengths]
            off = 0
            for b, n in enumerate(ns):
                if n:
                    sg.normal_bf16(raw_chunk[off:off + n], seed, synth.tensor_id(synth.RAW, li, b), c0 * D)
                    off += n
            layer.fill(layer.batch([min(L, c0 + n) if n else L for L, n in zip(lengths, ns)], ns), raw_chunk[:off])
        if layer.kind == "csa":
            bps = layer.cache.paging.max_blocks_per_seq
            n_ent = cap // m
            for b in range(S):
                r0 = b * bps * (128 // m)
                sg.e2m1_packed(layer.cache.keys.fp4[r0:r0 + n_ent], seed, synth.tensor_id(synth.IDX_K, li, b), 0)
                sg.ue8m0(layer.cache.keys.scale[r0:r0 + n_ent], seed, synth.tensor_id(synth.IDX_KS, li, b), 0)
    del raw_chunk
    # ---- per-step inputs of every layer (decode token L_b + s of every sequence)
    def gen(shape, dtype, fn, tid_kind, li, per_tok):
        t = torch.empty((steps_total, S) + shape, dtype=dtype, device=dev)
        for st in range(steps_total):
            for b in range(S):
                fn(t[st, b], seed, synth.tensor_id(tid_kind, li, b), (lengths[b] + st) * per_tok)
        return t
    raw_s, q_s, iq_s, iqs_s = [], [], [], []
    for li, layer in enumerate(stack.layers):
        raw_s.append(gen((D,), torch.bfloat16, sg.normal_bf16, synth.RAW, li, D))
        q_s.append(gen((H, D), torch.bfloat16, sg.normal_bf16, synth.QUERY, li, H * D))
        if layer.kind == "csa":
            iq_s.append(gen((Hi, r // 2), torch.uint8, sg.e2m1_packed, synth.IDX_Q, li, Hi * r))
            iqs_s.append(gen((Hi, r // 32), torch.uint8, sg.ue8m0, synth.IDX_QS, li, Hi * r // 32))
        else:
            iq_s.append(None)
            iqs_s.append(None)
    raw_in = [torch.empty((S, D), dtype=torch.bfloat16, device=dev) for _ in stack.layers]
    q_in = [torch.empty((S, H, D), dtype=torch.bfloat16, device=dev) for _ in stack.layers]
    iq_in = [torch.empty((S, Hi, r // 2), dtype=torch.uint8, device=dev) if x is not None else None for x in iq_s]
    iqs_in = [torch.empty((S, Hi, r // 32), dtype=torch.uint8, device=dev) if x is not None else None for x in iqs_s]
    hw_in = [torch.ones((S, Hi), dtype=torch.float32, device=dev) if x is not None else None for x in iq_s]
    outs = [torch.empty((S, H, D), dtype=torch.bfloat16, device=dev) for _ in stack.layers]
    cu_new = torch.arange(S + 1, dtype=torch.int32, device=dev)
    seq_len = torch.tensor([L + 1 for L in lengths], dtype=torch.int32, device=dev)
    batch = stack.layers[0].batch([cap] * S, [1] * S, cu_new=cu_new, seq_len=seq_len)
    base_len = torch.tensor(lengths, dtype=torch.int32, device=dev)

    def load_step(st):
        for li in range(n_layers):
            raw_in[li].copy_(raw_s[li][st]); q_in[li].copy_(q_s[li][st])
            if iq_in[li] is not None:
                iq_in[li].copy_(iq_s[li][st]); iqs_in[li].copy_(iqs_s[li][st])
        torch.add(base_len, st + 1, out=seq_len)

    def step_body():
        stack.step(batch, raw_in, q_in, outs, iq_in, iqs_in, hw_in)

    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    load_step(0)
    step_body()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph(keep_graph=True)
    with torch.cuda.graph(graph):
        step_body()
    graph.instantiate()
    graph_kernels = graph_kernel_count(graph)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps_total)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps_total)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for st in range(1, steps_total):
            load_step(st)
            flush.zero_()
            starts[st].record()
            graph.replay()
            ends[st].record()
        torch.cuda.synchronize()
    status_ok = all(v == 0 for v in stack.status)
    ms = statistics.mean(starts[st].elapsed_time(ends[st]) for st in range(args.warmup, steps_total))
    ms = max_over_ranks(ms, world, dev)
    # ---- whole-step algorithmic bytes (every layer is HBM-bound): CSA: 68 B per visible entry
    #      (indexer) + (k + 128) rows of 580 B; HCA: (visible entries + 128) rows of 580 B; both:
    #      query and output H x D BF16 per sequence
    row_b, key_b, qo_b = D - 64 + 128 + 4, r // 2 + r // 32, 2 * H * D * 2
    t_mid = args.warmup + args.steps // 2
    alg = 0
    for layer in stack.layers:
        for L in lengths:
            t = L + t_mid
            n = (t + 1) // layer.m
            if layer.kind == "csa":
                alg += n * key_b + (min(k, n) + min(t + 1, 128)) * row_b + qo_b
            else:
                alg += (n + min(t + 1, 128)) * row_b + qo_b
    hbm, peak_kind = measured_peaks()
    achieved = alg / (ms * 1e-3) / 1e9
    roofline = {"kernel": "whole step (every kernel of every layer)", "bound": "hbm", "achieved": round(achieved, 1),
                "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
                "algorithmic_bytes_per_launch": int(alg), "traffic": None}
    n_csa = sum(1 for kd in stack.kinds if kd == "csa")
    n_hca = n_layers - n_csa
    # CSA layer: compress (2) + indexer (2) + attention window part, top-k part, merge (3);
    # HCA layer: compress (2) + attention + merge (2)
    launches = n_csa * (2 + 1 + 3) + n_hca * (2 + 2)
    if graph_kernels is not None:   # counted from the captured step itself
        launches = graph_kernels
    cfg = {"workload": wl.name, "num_seqs": S, "layers": n_layers, "layer_kinds": stack.kinds,
           "ctx_len": lengths if wl.kind == "mixed" else wl.ctx_len, "new_tokens_per_seq": 1, "heads": H,
           "kv_dim": D, "row_format": "fp8_e4m3(448)+bf16_rope(64)+f32_scale", "csa_m": 4, "hca_m": 128,
           "top_k": k, "index_heads": Hi, "index_rank": r, "window": 128, "seed": wl.seed,
           "l2": "flushed between timed steps (256 MB write)", "data": "synthetic",
           "parallelism": f"replicas x{world} (independent sequences per GPU)"}
    return {"ms": ms, "clocks": clk.summary(), "roofline": roofline, "launches": launches,
            "status_ok": status_ok, "per_rank_queries": S, "config": cfg}


# ---------------------------------------------------------------------------------------------
# GPU arm, CSA prefill chunk: one sequence, 1M cached tokens + a chunk of new tokens (queries)
# ---------------------------------------------------------------------------------------------

def run_gpu_prefill(args, rank, world, local, wl):
    import torch
    import synth.gpu as sg
    import long_context_sparse_24_b300 as lcsa
    from long_context_sparse_24_b300.layer import Layer

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if lcsa.lcs_device_check() != 0:
        raise SystemExit("liblcsa needs a compute-capability 10.3 GPU")
    L, T, H, D = wl.ctx_len, wl.new_tokens, wl.heads, wl.dim
    Hi, r, k, m = wl.index_heads, wl.index_rank, wl.top_k, wl.m
    seed = rank_seed(wl.seed, rank)
    cap = L + T + 256
    layer = Layer("csa", 1, cap, H, D, lcsa.LCS_ROW_FP8_SPLIT, m, top_k=k, index_heads=Hi, index_rank=r,
                  max_new=T, device=dev)
    w = synth.bf16_bits_to_f32(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_W), 0, D)) / 16
    bias = synth.bf16_bits_to_f32(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_B), 0, 2 * m)) / 2
    layer.set_compressor(torch.from_numpy(w.astype(np.float32)).to(dev),
                         torch.from_numpy(bias.astype(np.float32)).to(dev))
    chunk = 65536
    raw = torch.empty((chunk, D), dtype=torch.bfloat16, device=dev)
    for c0 in range(0, L, chunk):
        n = min(chunk, L - c0)
        sg.normal_bf16(raw[:n], seed, synth.tensor_id(synth.RAW, 0, 0), c0 * D)
        layer.fill(layer.batch([c0 + n], [n]), raw[:n])
    n_ent = cap // m
    sg.e2m1_packed(layer.cache.keys.fp4[:n_ent], seed, synth.tensor_id(synth.IDX_K, 0, 0), 0)
    sg.ue8m0(layer.cache.keys.scale[:n_ent], seed, synth.tensor_id(synth.IDX_KS, 0, 0), 0)
    # the chunk's inputs: tokens L .. L+T-1
    raw_new = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
    sg.normal_bf16(raw_new, seed, synth.tensor_id(synth.RAW, 0, 0), L * D)
    q = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    sg.normal_bf16(q, seed, synth.tensor_id(synth.QUERY, 0, 0), L * H * D)
    iq = torch.empty((T, Hi, r // 2), dtype=torch.uint8, device=dev)
    sg.e2m1_packed(iq, seed, synth.tensor_id(synth.IDX_Q, 0, 0), L * Hi * r)
    iqs = torch.empty((T, Hi, r // 32), dtype=torch.uint8, device=dev)
    sg.ue8m0(iqs, seed, synth.tensor_id(synth.IDX_QS, 0, 0), L * Hi * r // 32)
    hw = torch.from_numpy(synth.head_weights(seed, synth.tensor_id(synth.HEAD_W, 0, 0), L * Hi, T * Hi)
                          .reshape(T, Hi).astype(np.float32)).to(dev)
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    batch = layer.batch([L + T], [T])

    def step_body():
        layer.step(batch, raw_new, q, out, idx_q_fp4=iq, idx_q_scale=iqs, head_w=hw)

    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    step_body()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph(keep_graph=True)
    with torch.cuda.graph(graph):
        step_body()
    graph.instantiate()
    graph_kernels = graph_kernel_count(graph)
    n_tot = args.warmup + args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_tot)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_tot)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for st in range(n_tot):
            flush.zero_()
            starts[st].record()
            graph.replay()
            ends[st].record()
        torch.cuda.synchronize()
    ms = statistics.mean(starts[st].elapsed_time(ends[st]) for st in range(args.warmup, n_tot))
    ms = max_over_ranks(ms, world, dev)
    # ---- per-stage device time: the step's calls one after another on one stream, untimed above
    cur = torch.cuda.current_stream()
    names = ["compress", "index_topk", "attend", "window_commit"]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
    stage = {n_: 0.0 for n_ in names}
    reps = 3
    for _ in range(reps):
        flush.zero_()
        ev[0].record(cur)
        layer.compress(batch, raw_new, cur); ev[1].record(cur)
        layer.select(batch, iq, iqs, hw, cur); ev[2].record(cur)
        layer.attend(batch, q, out, None, cur); ev[3].record(cur)
        layer.commit(batch, cur); ev[4].record(cur)
        torch.cuda.synchronize()
        for i_, n_ in enumerate(names):
            stage[n_] += ev[i_].elapsed_time(ev[i_ + 1]) / reps
    # ---- roofline of the dominant stage, a contraction: the indexer takes 2 r Hi FLOP per
    #      (query, visible entry) pair on FP8-class MMAs; the attention 4 H D FLOP per (query, row),
    #      rows = min(k, N(t)) + 128, on BF16/F16 MMAs
    pairs = sum((L + i + 1) // m for i in range(T))
    idx_flop = pairs * 2 * r * Hi
    att_flop = sum(4 * H * D * (min(k, (L + i + 1) // m) + 128) for i in range(T))
    peak_bf16 = None
    pth = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pth):
        peak_bf16 = json.load(open(pth)).get("bf16_tflops")
    peak_src = "of measured (MEASURED_PEAKS.json bf16_tflops)" if peak_bf16 else "of fallback"
    peak_bf16 = peak_bf16 or 1800.0
    if stage["index_topk"] >= stage["attend"]:
        kern, flop, t_ms, peak = ("index_tc_pf_kernel + topk_select_kernel (csa_index_topk)", idx_flop,
                                  stage["index_topk"], 2 * peak_bf16)
        peak_src += " x 2 (nominal FP8/BF16 ratio)"
    else:
        kern, flop, t_ms, peak = ("attend_tc_kernel (csa_attend: one CTA per query and 64-head group)", att_flop,
                                  stage["attend"], peak_bf16)
    achieved = flop / (t_ms * 1e-3) / 1e12
    roofline = {"kernel": kern, "bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1),
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "peak_source": peak_src,
                "flop_per_step": {"indexer": int(idx_flop), "attention": int(att_flop)},
                "stage_ms": {n_: round(v, 4) for n_, v in stage.items()}, "traffic": None}
    cfg = {"workload": wl.name, "num_seqs": 1, "ctx_len": L, "new_tokens_per_seq": T, "heads": H, "kv_dim": D,
           "row_format": "fp8_e4m3(448)+bf16_rope(64)+f32_scale", "m": m, "overlap": True, "index_heads": Hi,
           "index_rank": r, "index_format": "fp4_e2m1+ue8m0/32", "top_k": k, "window": 128, "seed": wl.seed,
           "step": "the same chunk of new tokens re-run every step (identical work)",
           "l2": "flushed between timed steps (256 MB write)", "data": "synthetic"}
    return {"ms": ms, "clocks": clk.summary(), "roofline": roofline, "status_ok": int(layer.status.item()) == 0,
            "per_rank_queries": T, "config": cfg,
            "launches": graph_kernels if graph_kernels is not None else 2 + 2 + 1 + 1}


# ---------------------------------------------------------------------------------------------
# GPU arm, indexer key production: block-scaled FP4 of the keys of a 1M-token CSA context
# ---------------------------------------------------------------------------------------------

def run_gpu_tensor_peak(args, rank, world, local):
    """The tensor-pipe rates the roofline fractions of the tensor-bound kernels are taken against:
    lcs_mma_probe, one CTA per SM issuing back-to-back tcgen05 MMAs of M = 128 (kind 0:
    kind::f8f6f4 with E2M1 operands, N = 256; kind 1: kind::f16, N = 256, the attention's MMA;
    kind 2: block-scaled kind::mxf4 with packed E2M1 operands, N = 240, the decode indexer's MMA),
    timed with CUDA events, best of the timed launches."""
    import torch
    import long_context_sparse_24_b300 as lcsa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if lcsa.lcs_device_check() != 0:
        raise SystemExit("liblcsa needs a compute-capability 10.3 GPU")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    mmas = 16384
    out = {}
    with ClockSampler(local) as clk:
        for kind, n_, kstep, name in ((0, 256, 32, "f8f6f4_e2m1"), (1, 256, 16, "f16"), (2, 240, 64, "mxf4_e2m1")):
            flop = 2.0 * 128 * n_ * kstep * mmas * sms
            times = []
            for it in range(args.warmup + args.steps):
                e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                lcsa.lcs_mma_probe(kind, mmas, sms, st)
                e1.record()
                torch.cuda.synchronize()
                if it >= args.warmup:
                    times.append(e0.elapsed_time(e1))
            out[name] = {"tflops": round(flop / (min(times) * 1e-3) / 1e12, 1),
                         "ms": round(min(times), 4), "flop_per_launch": flop}
    status_ok = int(st.item()) == 0
    return {"rates": out, "clocks": clk.summary(), "status_ok": status_ok, "sms": sms, "mmas": mmas}


def run_gpu_compress(args, rank, world, local):
    """csa_compress of a whole 1,048,576-token context of one sequence in one call (BF16 rows of
    D = 512 in, 262,144 entries of 580 B out, the window ring and pending rows updated), timed per
    call after an L2 flush.  Algorithmic bytes: the raw rows read once (1 GiB) and the entries
    written (152 MB); the overlapping windows re-read each block from L2/L1, not from HBM."""
    import torch
    import synth.gpu as sg
    import long_context_sparse_24_b300 as lcsa
    from long_context_sparse_24_b300.layer import Layer

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if lcsa.lcs_device_check() != 0:
        raise SystemExit("liblcsa needs a compute-capability 10.3 GPU")
    L, D, m = 1048576, 512, 4
    seed = rank_seed(7, rank)
    layer = Layer("csa", 1, L + 256, 64, D, lcsa.LCS_ROW_FP8_SPLIT, m, top_k=512, max_new=1, device=dev)
    w = synth.bf16_bits_to_f32(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_W), 0, D)) / 16
    bias = synth.bf16_bits_to_f32(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_B), 0, 2 * m)) / 2
    layer.set_compressor(torch.from_numpy(w.astype(np.float32)).to(dev),
                         torch.from_numpy(bias.astype(np.float32)).to(dev))
    raw = torch.empty((L, D), dtype=torch.bfloat16, device=dev)
    sg.normal_bf16(raw, seed, synth.tensor_id(synth.RAW, 0, 0), 0)
    batch = layer.batch([L], [L])
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    layer.fill(batch, raw)
    torch.cuda.synchronize()
    n_tot = args.warmup + args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_tot)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_tot)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for st in range(n_tot):
            flush.zero_()
            starts[st].record()
            layer.fill(batch, raw)       # the same context again: identical work and output
            ends[st].record()
        torch.cuda.synchronize()
    ms = statistics.mean(starts[st].elapsed_time(ends[st]) for st in range(args.warmup, n_tot))
    ms = max_over_ranks(ms, world, dev)
    hbm, peak_kind = measured_peaks()
    n_ent = L // m
    alg = L * D * 2 + n_ent * (D - 64 + 128 + 4)
    achieved = alg / (ms * 1e-3) / 1e9
    roofline = {"kernel": "compress_entries_kernel<512,1> + compress_state_kernel<512> (csa_compress)",
                "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                "algorithmic_bytes_per_launch": int(alg), "traffic": None}
    cfg = {"workload": "csa_compress_1m_d512_m4", "tokens": L, "dim": D, "m": m, "overlap": True,
           "entries": n_ent, "row_format": "fp8_e4m3(448)+bf16_rope(64)+f32_scale",
           "l2": "flushed between timed calls (256 MB write); input 1 GiB > L2", "data": "synthetic"}
    return {"ms": ms, "clocks": clk.summary(), "roofline": roofline, "per_rank_queries": L, "config": cfg,
            "launches": 2, "status_ok": int(layer.status.item()) == 0}


def run_gpu_attend_v(args, rank, world, local):
    """csa_attend with separate value rows on the decode shape of the headline (32 sequences of
    131,072 tokens, one query each, 64 heads, D = 512 FP8-split rows, k = 512 selected entries of
    32,768 plus the 128-row window), timed per call after an L2 flush; the shared-KV call on the
    same rows is timed beside it.  Key and value rows are random codes, RoPE dims and scales;
    each query's selection is a random sorted set of visible entries.  Algorithmic bytes per
    query: (k + 128) key rows and as many value rows of 580 B, the query and the output."""
    import torch
    import synth.gpu as sg
    import long_context_sparse_24_b300 as lcsa
    from long_context_sparse_24_b300 import buffers

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if lcsa.lcs_device_check() != 0:
        raise SystemExit("liblcsa needs a compute-capability 10.3 GPU")
    S, L, H, D, m, k = 32, 131072, 64, 512, 4, 512
    seed = rank_seed(9, rank)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    fmt = lcsa.LCS_ROW_FP8_SPLIT
    cache = buffers.alloc_layer(S, L, D, fmt, m, True, 0, dev)

    def fill(rows, tid):
        n = rows.nope.shape[0]
        codes = torch.randint(0, 0x7E, rows.nope.shape, dtype=torch.int32, device=dev, generator=gen)
        sign = torch.randint(0, 2, rows.nope.shape, dtype=torch.int32, device=dev, generator=gen) << 7
        rows.nope.copy_((codes | sign).to(torch.uint8))
        sg.normal_bf16(rows.rope, seed, synth.tensor_id(tid), 0)
        rows.scale.copy_(0.01 + 0.001 * torch.rand(n, device=dev, generator=gen))

    values = lcsa.Values(buffers.alloc_rows(fmt, D, cache.entries.num_rows, dev),
                         buffers.alloc_rows(fmt, D, cache.state.window.num_rows, dev))
    for rows, tid in ((cache.entries, synth.RAW), (cache.state.window, synth.RAW),
                      (values.entries, synth.QUERY), (values.window, synth.QUERY)):
        fill(rows, tid)
    n_vis = L // m
    idx = torch.stack([torch.sort(torch.randperm(n_vis, device=dev, generator=gen)[:k]).values
                       for _ in range(S)]).to(torch.int32)
    cnt = torch.full((S,), k, dtype=torch.int32, device=dev)
    q = torch.empty((S, H, D), dtype=torch.bfloat16, device=dev)
    sg.normal_bf16(q, seed, synth.tensor_id(synth.QUERY), 0)
    batch = buffers.make_batch([L] * S, [1] * S, dev)
    out = torch.empty((S, H, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((S, H), dtype=torch.float32, device=dev)
    wsb = lcsa.lcs_attend_workspace(batch, H, D, k + 128)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = 1 / math.sqrt(D)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def one_call(v):
        lcsa.csa_attend(batch, q, H, idx, cnt, k, m, cache.entries, cache.paging, cache.state, scale, out, lse, ws,
                        wsb, status, values=v)

    def two_calls():   # the decode step's form: window part, then the top-k part and the merge
        lcsa.csa_attend_window(batch, q, H, k, m, cache.entries, cache.paging, cache.state, scale, ws, wsb, status)
        lcsa.csa_attend_topk(batch, q, H, idx, cnt, k, m, cache.entries, cache.paging, cache.state, scale, out, lse,
                             ws, wsb, status)

    # each form captured once (the timed launches carry no host marshalling)
    graphs = {}
    for name, fn in (("separate_v", lambda: one_call(values)), ("shared_kv", lambda: one_call(None)),
                     ("shared_kv_two_calls", two_calls)):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs[name] = g
    n_tot = args.warmup + args.steps
    times = {}
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for name, g in graphs.items():
            starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_tot)]
            ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_tot)]
            for st in range(n_tot):
                flush.zero_()
                starts[st].record()
                g.replay()
                ends[st].record()
            torch.cuda.synchronize()
            times[name] = statistics.mean(starts[st].elapsed_time(ends[st]) for st in range(args.warmup, n_tot))
    ms = max_over_ranks(times["separate_v"], world, dev)
    hbm, peak_kind = measured_peaks()
    row = D - 64 + 128 + 4
    alg = S * ((k + 128) * row * 2 + 2 * H * D * 2)
    achieved = alg / (ms * 1e-3) / 1e9
    roofline = {"kernel": "attend_kernel<512, FP8_SPLIT, 4, separate values> + attend_combine_kernel (csa_attend)",
                "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                "algorithmic_bytes_per_launch": int(alg), "traffic": None}
    cfg = {"workload": "csa_attend_separate_v_32x128k", "num_seqs": S, "ctx_len": L, "heads": H, "kv_dim": D,
           "top_k": k, "window": 128, "row_format": "fp8_e4m3(448)+bf16_rope(64)+f32_scale, keys and values apart",
           "shared_kv_ms": round(times["shared_kv"], 5), "shared_kv_two_calls_ms": round(times["shared_kv_two_calls"], 5),
           "timing": "one CUDA graph replay per timed call",
           "l2": "flushed between timed calls (256 MB write)", "data": "synthetic"}
    return {"ms": ms, "clocks": clk.summary(), "roofline": roofline, "per_rank_queries": S, "config": cfg,
            "launches": 2, "status_ok": int(status.item()) == 0}


def run_gpu_sink(args, rank, world, local):
    """lcs_attention_sink over the attention outputs of the CSA prefill chunk (16,384 queries x 128
    heads x 512 dims BF16, 2.1 GB: far beyond L2), timed per launch after an L2 flush."""
    import torch
    import synth.gpu as sg
    import long_context_sparse_24_b300 as lcsa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if lcsa.lcs_device_check() != 0:
        raise SystemExit("liblcsa needs a compute-capability 10.3 GPU")
    T, H, D = 16384, 128, 512
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    sg.normal_bf16(out, rank_seed(6, rank), synth.tensor_id(synth.QUERY), 0)
    lse = torch.full((T, H), 3.0, dtype=torch.float32, device=dev)
    sink = torch.linspace(-2.0, 2.0, H, dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    n_tot = args.warmup + args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_tot)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_tot)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for st in range(n_tot):
            flush.zero_()
            starts[st].record()
            lcsa.lcs_attention_sink(out, lse, sink)
            ends[st].record()
        torch.cuda.synchronize()
    ms = statistics.mean(starts[st].elapsed_time(ends[st]) for st in range(args.warmup, n_tot))
    ms = max_over_ranks(ms, world, dev)
    hbm, peak_kind = measured_peaks()
    alg = T * H * (2 * D * 2 + 8)
    achieved = alg / (ms * 1e-3) / 1e9
    roofline = {"kernel": "attention_sink_kernel (lcs_attention_sink)", "bound": "hbm", "achieved": round(achieved, 1),
                "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)", "algorithmic_bytes_per_launch": alg,
                "traffic": None}
    cfg = {"workload": "attention_sink_16384q_h128_d512", "queries": T, "heads": H, "dim": D,
           "l2": "flushed between timed launches (256 MB write); outputs 2.1 GB > L2", "data": "synthetic"}
    return {"ms": ms, "clocks": clk.summary(), "roofline": roofline, "per_rank_queries": T, "config": cfg,
            "launches": 1}


def run_gpu_quantize(args, rank, world, local):
    """lcs_quantize_e2m1 over 4 x 266,240 BF16 rows of rank 128 (the indexer keys of a 1M-token
    CSA context in four layers: more than L2), timed per launch after an L2 flush."""
    import torch
    import synth.gpu as sg
    import long_context_sparse_24_b300 as lcsa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if lcsa.lcs_device_check() != 0:
        raise SystemExit("liblcsa needs a compute-capability 10.3 GPU")
    rows, r = 4 * 266240, 128
    x = torch.empty((rows, r), dtype=torch.bfloat16, device=dev)
    sg.normal_bf16(x, rank_seed(5, rank), synth.tensor_id(synth.IDX_K), 0)
    codes = torch.empty((rows, r // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((rows, r // 32), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    n_tot = args.warmup + args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_tot)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_tot)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for st in range(n_tot):
            flush.zero_()
            starts[st].record()
            lcsa.lcs_quantize_e2m1(x, codes, scales)
            ends[st].record()
        torch.cuda.synchronize()
    ms = statistics.mean(starts[st].elapsed_time(ends[st]) for st in range(args.warmup, n_tot))
    ms = max_over_ranks(ms, world, dev)
    hbm, peak_kind = measured_peaks()
    alg = rows * (r * 2 + r // 2 + r // 32)
    achieved = alg / (ms * 1e-3) / 1e9
    roofline = {"kernel": "quantize_e2m1_kernel (lcs_quantize_e2m1)", "bound": "hbm", "achieved": round(achieved, 1),
                "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)", "algorithmic_bytes_per_launch": alg,
                "traffic": None}
    cfg = {"workload": "index_keys_fp4_4x266240_r128", "rows": rows, "rank": r, "input": "bf16 rows",
           "output": "fp4_e2m1 codes + ue8m0 per 32", "l2": "flushed between timed launches (256 MB write); "
           "input 273 MB > L2", "data": "synthetic"}
    return {"ms": ms, "clocks": clk.summary(), "roofline": roofline, "status_ok": True, "per_rank_queries": rows,
            "config": cfg, "launches": 1}


def run_e2e(torch, layer, batch, graph, raw_in, q_in, iq_in, iqs_in, hw_in, out, seq_len, raw_steps, q_steps,
            iq_steps, iqs_steps, hw_steps, args, L, S, flush):
    """Same step with its inputs copied from pinned host memory and the output read back, all
    inside one CUDA graph: the small inputs (new KV rows, indexer queries, lengths) first on the
    step's stream; the attention queries on a copy stream that only the attention waits for, so
    that the largest copy runs next to compression and the indexer; the output copied back at
    the end.  Before each replay the host writes that step's inputs into the pinned staging
    buffers the graph copies from (outside the timed region, as a producer of the inputs would)."""
    import long_context_sparse_24_b300 as lcsa
    n = min(args.steps, 8)
    host_in = [t[:n].cpu() for t in (raw_steps, q_steps, iq_steps, iqs_steps, hw_steps)]
    stage = [torch.empty(t.shape[1:], dtype=t.dtype).pin_memory() for t in host_in]
    seq_host = torch.empty(seq_len.shape, dtype=torch.int32).pin_memory()
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in stage) + seq_host.numel() * 4
    d2h = out.numel() * out.element_size()
    main = torch.cuda.Stream()
    copy = torch.cuda.Stream()
    q_ready = torch.cuda.Event()

    def body():
        # host -> device through lcs_stage_copy (kernels reading the pinned pages; the copy engine
        # moves MB-sized host inputs several times slower); device -> host by the copy engine
        copy.wait_stream(main)
        lcsa.lcs_stage_copy([(q_in, stage[1])], stream=copy)
        q_ready.record(copy)
        lcsa.lcs_stage_copy([(raw_in, stage[0]), (iq_in, stage[2]), (iqs_in, stage[3]), (hw_in, stage[4]),
                             (seq_len, seq_host)], stream=main)
        layer.step(batch, raw_in, q_in, out, idx_q_fp4=iq_in, idx_q_scale=iqs_in, head_w=hw_in, stream=main,
                   q_ready=q_ready)
        host_out.copy_(out, non_blocking=True)
        main.wait_stream(copy)

    # rewind the state positions: re-run decode positions L+warmup+steps .. (new tokens, same shapes)
    base = L + args.warmup + args.steps + 5
    seq_host.fill_(base)
    for k_, t in enumerate(host_in):
        stage[k_].copy_(t[0])
    torch.cuda.synchronize()
    main.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(main):
        body()                          # eager once (the copy stream and events warm up)
    main.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        body()
    times, host_times = [], []
    for s in range(n):
        for k_, t in enumerate(host_in):
            stage[k_].copy_(t[s])
        seq_host.fill_(base + s + 1)
        flush.zero_()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(main):
            h0 = time.perf_counter()
            e0.record(main)
            g.replay()
            e1.record(main)
        main.synchronize()
        host_times.append((time.perf_counter() - h0) * 1e3)
        times.append(e0.elapsed_time(e1))
    ms = statistics.mean(times)
    host_ms = statistics.mean(host_times)
    return {"value": round(S / (ms * 1e-3), 1), "unit": UNIT, "ms_per_step": round(ms, 4),
            "host_clock": {"value": round(S / (host_ms * 1e-3), 1), "ms_per_step": round(host_ms, 4),
                           "timing": "host perf_counter from before the replay to after the stream synchronise"},
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": n,
            "api": "Layer.step (csa_compress, csa_attend_window | csa_index_topk, csa_attend_topk) with the "
                   "host copies, one CUDA graph per step"}


# ---------------------------------------------------------------------------------------------
# oracle (CPU) arm
# ---------------------------------------------------------------------------------------------

class OracleDecode:
    """The fp64 oracle serving decode steps of a few workload sequences."""

    def __init__(self, n_seqs: int, seed: int):
        import oracle
        self.o = oracle
        D, m, r, Hi = WL.dim, WL.m, WL.index_rank, WL.index_heads
        self.w = (synth.bf16_bits_to_f32(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_W), 0, D)) / 16).astype(np.float64)
        self.bias = (synth.bf16_bits_to_f32(synth.normal_bf16(seed, synth.tensor_id(synth.COMP_B), 0, 2 * m)) / 2).astype(np.float64)
        self.seed = seed
        self.seqs = []
        L = WL.ctx_len
        for b in range(n_seqs):
            raw = synth.bf16_bits_to_f32(synth.normal_bf16(seed, synth.tensor_id(synth.RAW, 0, b), 0, (L + 64) * D))
            raw = raw.reshape(L + 64, D).astype(np.float64)
            ent = oracle.quantize_rows(oracle.compress_blocked(raw[:L], self.w, self.bias, m, True), "fp8_split")["deq"]
            win = oracle.quantize_rows(raw[L - 128:L], "fp8_split")["deq"]
            n_ent = (L + 64) // m
            kc = synth.e2m1_codes(seed, synth.tensor_id(synth.IDX_K, 0, b), 0, n_ent * r).reshape(n_ent, r)
            ks = synth.ue8m0_scales(seed, synth.tensor_id(synth.IDX_KS, 0, b), 0, n_ent * r // 32).reshape(n_ent, r // 32)
            self.seqs.append({"raw": raw, "ent": list(ent), "win": list(win), "t": L, "kc": kc, "ks": ks})

    def step(self, b: int):
        """Decode the next token of sequence b: compress, index + top-k, attend."""
        o, s = self.o, self.seqs[b]
        D, H, m, r, Hi, k = WL.dim, WL.heads, WL.m, WL.index_rank, WL.index_heads, WL.top_k
        t = s["t"]
        if (t + 1) % m == 0:
            e = o.compress(s["raw"][:t + 1], self.w, self.bias, m, True, (t + 1) // m - 1, 1)
            s["ent"].append(o.quantize_rows(e, "fp8_split")["deq"][0])
        s["win"].append(o.quantize_rows(s["raw"][t:t + 1], "fp8_split")["deq"][0])
        s["win"] = s["win"][-128:]
        qc = synth.e2m1_codes(self.seed, synth.tensor_id(synth.IDX_Q, 0, b), t * Hi * r, Hi * r).reshape(1, Hi, r)
        qs = synth.ue8m0_scales(self.seed, synth.tensor_id(synth.IDX_QS, 0, b), t * Hi * r // 32, Hi * r // 32)
        hw = synth.head_weights(self.seed, synth.tensor_id(synth.HEAD_W, 0, b), t * Hi, Hi).reshape(1, Hi)
        n = o.visible_entries(t, m)
        sc = o.index_scores(qc, qs.reshape(1, Hi, r // 32), hw, s["kc"][:n], s["ks"][:n])
        sel = o.topk_select(sc[0], k)
        q = synth.bf16_bits_to_f32(synth.normal_bf16(self.seed, synth.tensor_id(synth.QUERY, 0, b), t * H * D, H * D))
        rows = np.concatenate([np.asarray(s["ent"])[sel], np.asarray(s["win"])])
        out, _ = o.attend(q.reshape(H, D).astype(np.float64), rows, 1 / math.sqrt(D))
        s["t"] = t + 1
        return out


def oracle_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(budget_s: float = 12.0, n_seqs: int = 2):
    od = OracleDecode(n_seqs, WL.seed)
    done, t0 = 0, time.perf_counter()
    while True:
        od.step(done % n_seqs)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or done >= 400:
            break
    return {"value": round(done / el, 3), "unit": UNIT, "cores": oracle_cores(), "kind": "oracle",
            "sample": f"{done} decode queries of {n_seqs} workload sequences (131072-token contexts; cache "
                      f"built untimed), fp64 numpy oracle, {el:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    od = OracleDecode(2, WL.seed)
    for i in range(args.warmup):
        od.step(i % 2)
    times = []
    per_step = 2                     # bounded sample: 2 decode queries per step
    for s in range(args.steps):
        t0 = time.perf_counter()
        for b in range(per_step):
            od.step(b)
        times.append(time.perf_counter() - t0)
    ms = statistics.mean(times) * 1e3
    val = per_step / (ms * 1e-3)
    cores = oracle_cores()
    return {"metric": METRIC, "value": round(val, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_config({"sample_per_step": f"{per_step} decode queries"}),
            "cpu_baseline": {"value": round(val, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} decode queries per step of 2 workload sequences"},
            "e2e": {"value": round(val, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line))
        return
    assert args.warmup >= 3, "at least 3 warm-up steps"
    if args.workload == "tensor_peak":
        res = run_gpu_tensor_peak(args, rank, world, local)
        if rank == 0:
            r = res["rates"]
            print(json.dumps({"metric": "tcgen05 tensor-pipe rate (probe): block-scaled FP4", "value": r["mxf4_e2m1"]["tflops"],
                              "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "ms_per_step": r["mxf4_e2m1"]["ms"], "higher_is_better": True, "scaling": "weak",
                              "vs_baseline": None, "dtype": "e2m1 x e2m1 (ue8m0 per 32) -> f32 (kind::mxf4)",
                              "data": "synthetic",
                              "config": {"workload": "tcgen05_mma_probe_m128", "ctas": res["sms"],
                                         "mmas_per_cta": res["mmas"], "timing": "best of the timed launches"},
                              "rates": r, "clocks": res["clocks"], "e2e": None,
                              "gpu_launches": 3 * (args.warmup + args.steps), "device_status_ok": res["status_ok"]}))
        return
    if args.workload == "compress_1m":
        res = run_gpu_compress(args, rank, world, local)
        if rank == 0:
            print(json.dumps({"metric": "raw KV tokens compressed per second (CSA, m = 4, overlapping)",
                              "value": round(job_value(res["per_rank_queries"], world, res["ms"]), 1),
                              "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "ms_per_step": round(res["ms"], 5), "higher_is_better": True, "scaling": "weak",
                              "vs_baseline": None, "dtype": "bf16 in, fp8 e4m3 + bf16 rope + f32 scale out, fp32 math",
                              "data": "synthetic", "config": res["config"], "roofline": res["roofline"],
                              "clocks": res["clocks"], "e2e": None, "gpu_launches": res["launches"] * args.steps,
                              "device_status_ok": res["status_ok"]}))
        return
    if args.workload not in ("csa_decode", "csa_decode_1m"):
        if args.workload == "attend_separate_v":
            res = run_gpu_attend_v(args, rank, world, local)
            if rank == 0:
                print(json.dumps({"metric": METRIC, "value": round(job_value(res["per_rank_queries"], world, res["ms"]), 1),
                                  "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                                  "ms_per_step": round(res["ms"], 5), "higher_is_better": True, "scaling": "weak",
                                  "vs_baseline": None, "dtype": "fp8 e4m3 + bf16 rows, bf16 queries, fp32 softmax",
                                  "data": "synthetic", "config": res["config"], "roofline": res["roofline"],
                                  "clocks": res["clocks"], "e2e": None,
                                  "gpu_launches": res["launches"] * args.steps, "device_status_ok": res["status_ok"]}))
            return
        if args.workload == "attention_sink":
            res = run_gpu_sink(args, rank, world, local)
            if rank == 0:
                print(json.dumps({"metric": METRIC, "value": round(job_value(res["per_rank_queries"], world, res["ms"]), 1),
                                  "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                                  "ms_per_step": round(res["ms"], 5), "higher_is_better": True, "scaling": "weak",
                                  "vs_baseline": None, "dtype": "bf16 outputs, fp32 lse", "data": "synthetic",
                                  "config": res["config"], "roofline": res["roofline"], "clocks": res["clocks"],
                                  "e2e": None, "gpu_launches": res["launches"] * args.steps, "device_status_ok": True}))
            return
        if args.workload == "index_key_quantize":
            res = run_gpu_quantize(args, rank, world, local)
            if rank == 0:
                print(json.dumps({"metric": "indexer key rows quantised to block-scaled FP4 per second",
                                  "value": round(job_value(res["per_rank_queries"], world, res["ms"]), 1),
                                  "unit": "rows/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                                  "ms_per_step": round(res["ms"], 5), "higher_is_better": True, "scaling": "weak",
                                  "vs_baseline": None, "dtype": "bf16 in, fp4 e2m1 + ue8m0 out", "data": "synthetic",
                                  "config": res["config"], "roofline": res["roofline"], "clocks": res["clocks"],
                                  "e2e": None, "gpu_launches": res["launches"] * args.steps, "device_status_ok": True}))
            return
        runner = run_gpu_prefill if args.workload == "csa_prefill" else run_gpu_stack
        wl = synth.CONFIGS[args.workload]
        if args.workload == "csa_prefill" and (args.ctx_len is not None or args.new_tokens is not None):
            import dataclasses
            ctx = args.ctx_len if args.ctx_len is not None else wl.ctx_len
            new_ = args.new_tokens if args.new_tokens is not None else wl.new_tokens
            wl = dataclasses.replace(wl, name=f"csa_prefill_{ctx}_plus_{new_}_h{wl.heads}_d{wl.dim}", ctx_len=ctx,
                                     new_tokens=new_)
        res = runner(args, rank, world, local, wl)
        if rank == 0:
            value = job_value(res["per_rank_queries"], world, res["ms"])
            print(json.dumps({"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
                              "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["ms"], 5),
                              "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                              "dtype": "fp8/fp4 storage, f16/bf16 MMA, fp32 accumulate", "data": "synthetic",
                              "config": res["config"], "roofline": res["roofline"], "clocks": res["clocks"],
                              "e2e": None, "gpu_launches": res["launches"] * args.steps,
                              "device_status_ok": res["status_ok"]}))
        return
    wl = synth.CONFIGS[args.workload]
    if args.num_seqs is not None:
        import dataclasses
        wl = dataclasses.replace(wl, name=wl.name.replace(f"{wl.num_seqs}x", f"{args.num_seqs}x", 1),
                                 num_seqs=args.num_seqs)
    res = run_gpu(args, rank, world, local, wl)
    if rank == 0:
        value = job_value(res["per_rank_queries"], world, res["ms"])
        line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(res["ms"], 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "fp8/fp4 storage, bf16/f16 MMA, fp32 accumulate",
                "data": "synthetic",
                "config": workload_config(wl=wl, extra={"parallelism": f"replicas x{world} (independent sequences per GPU)",
                                           "stage_ms_source": "separate replays of a serialised copy of the step with event nodes between calls (the timed step runs compress and attend_window next to index_topk)",
                                           "stage_ms": {k_: round(v, 5) for k_, v in res["stages"].items()}}),
                "roofline": res["roofline"], "roofline_other": res["roofline_other"],
                "roofline_step": res["roofline_step"], "clocks": res["clocks"],
                "e2e": res["e2e"],
                "gpu_launches": res["launches"], "device_status_ok": res["status_ok"]}
        if not args.no_cpu_baseline and world == 1 and wl is WL:
            line["cpu_baseline"] = cpu_baseline()
        if world == 1 and wl is WL and args.others != "none":
            line["other_workloads"] = run_others(args)
        print(json.dumps(line))


if __name__ == "__main__":
    main()
