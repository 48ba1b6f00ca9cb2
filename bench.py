"""Benchmark of the CSA2 attention step on GB300.

Default workload: FULL-layer decode batch -- 64 sequences with context lengths
uniform in [16384, 65536], ratio 2 (compressor with odd-tail state), 64-head x
128-d indexer over the visible rows, top-512, 64 x 512 queries over the 128-slot
bf16 window plus the selected rows with a per-head sink.  One step = compress the
64 new tokens + index + top-512 + sparse attention, all through the C ABI.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle instead.
Under torchrun every rank runs its own batch (weak scaling, no collective on the
data path); the step time is the maximum over ranks.
"""
import argparse
import copy
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA2 decode queries/sec & achieved HBM GB/s (index+top-512+sparse_attn), 1 GB300"
PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="decode",
                    choices=["tiny", "decode", "reindex", "prefill", "long", "prefill_small",
                             "reindex_small", "long_small"],
                    help="workload; the *_small ones are reduced cases for profiler captures")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-queries", type=int, default=64)
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the REINDEX / prefill / long figures of the default line")
    ap.add_argument("--stages", action="store_true",
                    help="time every entry point of the step (and the candidate-pool and "
                         "inverse-RoPE variants) on its own instead; prints one JSON line")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, world, device):
    """The largest value of x over the ranks (x itself on one rank)."""
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_value(units_per_rank, world, steps, ms_max):
    """Whole-job throughput of a weak-scaling run: the units every rank processed in
    `steps` steps over the slowest rank's time (ms)."""
    return units_per_rank * world * steps / (ms_max / 1e3)


def hbm_peak():
    try:
        with open(PEAKS) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM, "fallback"


def make_workload(name, rank):
    from synth import workloads as W
    seed_off = 1000 * rank
    if name == "decode":
        return W.decode_batch(seed=1 + seed_off)
    if name == "tiny":
        return W.tiny_decode(seed=0 + seed_off)
    if name == "reindex":
        return W.reindex_decode(seed=2 + seed_off)
    if name == "prefill":
        return W.prefill_reuse(seed=3 + seed_off)
    # reduced cases of the same shapes (inputs still larger than L2) for profiler captures
    if name == "prefill_small":
        return W.prefill_reuse(n_new=512, layers=1, seed=3 + seed_off)
    if name == "reindex_small":
        return W.reindex_decode(ctx=32768, seed=2 + seed_off)
    if name == "long_small":
        return W.long_decode(ctx=131072, seed=4 + seed_off)
    return W.long_decode(seed=4 + seed_off)


def spec_for(wl):
    from csa2_compressed_sparse_gb300 import SWA_LINEAR, SWA_RING
    from csa2_compressed_sparse_gb300.step import StepSpec
    ms = wl.ncb * 8 if wl.reindex else int(max((int(p) + 1) // wl.ratio for p in wl.q_pos))
    return StepSpec(ratio=wl.ratio, H=wl.H, k=wl.k, max_scored=ms,
                    swa_mode=SWA_LINEAR if wl.swa == "linear" else SWA_RING)


def algorithmic_bytes(wl):
    """Bytes a step must move at least (the scores spill is excluded).
    Returns (total, index-stage bytes, attention bytes per layer)."""
    nvis = np.array([(int(p) + 1) // wl.ratio for p in wl.q_pos], dtype=np.int64)
    scored = np.full_like(nvis, wl.ncb * 8) if wl.reindex else nvis
    keff = np.minimum(scored, wl.k)
    index = int((scored * 128 * 2).sum()) + wl.Q * (wl.H * 128 * 2 + wl.H * 4 + wl.k * 4)
    if wl.reindex:
        index += wl.Q * wl.ncb * 4
    win_row = 528 if wl.swa_dtype == "fp8" else 1024
    win = np.minimum(wl.q_pos + 1, 128)
    if wl.swa == "linear":  # windows of neighbouring queries overlap: count the distinct rows
        win_bytes = int(wl.lin_len.sum()) * 1024
    else:
        win_bytes = int(win.sum()) * win_row
    attn = int(keff.sum()) * 1024 + win_bytes + wl.Q * (64 * 512 * 2 * 2 + wl.k * 4 + 64)
    comp = wl.T * 512 * 2 * 2 + int((wl.n_rows - wl.n_hist).sum()) * 1024 + wl.B * 2 * 512 * 4 * 2
    return comp + index + attn * wl.layers, index, attn


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def steps_per_graph(steps, cap=32):
    """Steps captured in one CUDA graph: the largest divisor of `steps` up to `cap`."""
    return max(g for g in range(1, min(cap, max(steps, 1)) + 1) if steps % g == 0)


def upload_graphs(graphs, stream):
    """Upload instantiated graphs to the device (cuGraphUpload), so that their first replay
    costs no more than any other; where the exec handle is not exposed, replay each once."""
    import ctypes
    try:
        cu = ctypes.CDLL("libcuda.so.1")
        cu.cuGraphUpload.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        for g in graphs:
            if cu.cuGraphUpload(ctypes.c_void_p(g.raw_cuda_graph_exec()),
                                ctypes.c_void_p(stream.cuda_stream)) != 0:
                raise RuntimeError("cuGraphUpload failed")
    except (AttributeError, OSError, RuntimeError):
        for g in graphs:
            g.replay()
    torch.cuda.synchronize()


def step_fn(csa2, spec, t, buf, side_c, fused=True):
    """One step on the current stream, returned as a function of an optional pair of
    events recorded around the index stage.  fused: the compressor's tokens run inside
    the indexer's call (csa2_compress_index_topk), so the whole step is one chain of
    kernels on one stream.  Otherwise csa2_compress runs on `side_c`, concurrently with
    index + top-k (it writes only the main plane, which the indexer does not read), and
    is joined before the attention."""
    from csa2_compressed_sparse_gb300.step import swa_of

    def one_step(ev=None):
        cur = torch.cuda.current_stream()
        comp = t["kv"].shape[0] > 0
        if not fused:
            side_c.wait_stream(cur)
            with torch.cuda.stream(side_c):
                if comp:
                    csa2.csa2_compress(t["kv"], t["score"], t["cu_seqlens"], t["start_pos"],
                                       spec.ratio, t["kv_state"], t["score_state"], t["plane"],
                                       t["row_base"], t["inv_freq"], eps=spec.eps)
        if ev is not None:
            ev[0].record()
        if fused and comp:
            csa2.csa2_compress_index_topk(
                t["kv"], t["score"], t["cu_seqlens"], t["start_pos"], t["kv_state"],
                t["score_state"], t["plane"], t["inv_freq"], t["iq"], t["w"], t["index_k"],
                t["row_base"], t["q_seq"], t["q_pos"], spec.ratio, spec.k, spec.max_scored,
                buf.sel, buf.ws, sel_scores=buf.sel_scores, cand=t.get("cand"),
                relu=spec.relu, eps=spec.eps)
        else:
            csa2.csa2_index_topk(t["iq"], t["w"], t["index_k"], t["row_base"], t["q_seq"],
                                 t["q_pos"], spec.ratio, spec.k, spec.max_scored, buf.sel,
                                 buf.ws, sel_scores=buf.sel_scores, cand=t.get("cand"),
                                 relu=spec.relu)
        if ev is not None:
            ev[1].record()
        if not fused:
            cur.wait_stream(side_c)
        for layer in range(len(t["q"])):
            fn = csa2.csa2_sparse_attn if layer == 0 else csa2.csa2_reuse_attn
            fn(t["q"][layer], t["q_seq"], t["q_pos"], swa_of(spec, t, layer), t["plane"],
               t["row_base"], buf.sel, t["sink"], buf.out[layer], scale=spec.scale,
               ws=buf.attn_ws)

    return one_step


def traffic_from_profile(config):
    """DRAM bytes per launch of the index score kernel from the committed ncu summary."""
    p = os.path.join(ROOT, "profiles", f"index_score_kernel.{config}.md")
    try:
        for line in open(p):
            if line.startswith("dram_bytes_per_launch:"):
                v = line.split(":", 1)[1].strip()
                return None if v == "null" else float(v)
    except OSError:
        pass
    return None


def run_ours(args):
    import torch.distributed as dist
    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    import csa2_compressed_sparse_gb300 as csa2
    from csa2_compressed_sparse_gb300.step import allocate, kernel_launches, run_step

    wl = make_workload(args.config, rank)
    spec = spec_for(wl)
    t = wl.materialize("cuda")
    buf = allocate(spec, t)
    stream = torch.cuda.current_stream()
    run_step(spec, t, buf)
    csa2.csa2_device_status()

    # ---- device-resident timing of K steps ----
    # The K steps run as replays of CUDA graphs that each hold G consecutive steps (G the
    # largest divisor of K up to 32; the C ABI only enqueues kernels, so it captures as is):
    # inside a graph the kernels of one step follow those of the previous step with
    # programmatic dependent launch, as they would in an engine's decode loop, instead of
    # paying a graph launch per step.  Every step keeps its full order: a step's first
    # kernels wait for the previous step's last one.  The index stage is timed on the
    # launching stream by event-record nodes: NS copies of the G-step graph carry a pair of
    # events around the index stage of their middle step and replace every (K/G // NS)-th
    # plain replay, so the sampled durations span the timed region without a host
    # synchronisation inside it.  Every graph is uploaded to the device before the
    # warm-up, so no replay in the timed region pays for its first launch.
    side_c = torch.cuda.Stream()
    one_step = step_fn(csa2, spec, t, buf, side_c)

    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        one_step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    G = steps_per_graph(args.steps)
    n_chain = args.steps // G
    n_samples = max(1, min(n_chain, 32))
    stride = n_chain // n_samples
    sample_ev = [(torch.cuda.Event(enable_timing=True, external=True),
                  torch.cuda.Event(enable_timing=True, external=True))
                 for _ in range(n_samples)]

    def capture(n, ev=None):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                one_step(ev if i == n // 2 else None)
        return g

    g_one = capture(1)                 # warm-up steps
    g_plain = capture(G)
    g_sample = [capture(G, ev) for ev in sample_ev]
    upload_graphs([g_one, g_plain] + g_sample, stream)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    # the W warm-up steps run after the clock sampler's start-up pause, so that the GPU
    # enters the timed region from the warm-up, not from idle
    for i in range(max(args.warmup, 3)):
        g_one.replay()
    torch.cuda.synchronize()
    csa2.csa2_device_status()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for i in range(n_chain):
        j, r = divmod(i, stride)
        (g_sample[j] if r == 0 and j < n_samples else g_plain).replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    ms = ev0.elapsed_time(ev1)
    idx_ms = sum(a.elapsed_time(b) for a, b in sample_ev) / n_samples
    csa2.csa2_device_status()
    ms = max_over_ranks(ms, world, "cuda")
    ms_step = ms / args.steps
    value = weak_value(wl.Q, world, args.steps, ms)
    total_bytes, index_bytes, attn_bytes = algorithmic_bytes(wl)
    # the index stage is the csa2_compress_index_topk call: the compressor's bytes are in it
    index_bytes += total_bytes - index_bytes - attn_bytes * wl.layers
    peak, peak_kind = hbm_peak()
    achieved_index = index_bytes / (idx_ms / 1e3) / 1e9

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, wl, spec, t, buf, world, ms_step)

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "queries/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64 generator, N(0,1)-like values)",
        "config": {
            "workload": wl.name,
            "description": wl.description,
            "queries_per_step_per_gpu": wl.Q,
            "sequences": wl.B,
            "ratio": wl.ratio,
            "indexer_heads": wl.H,
            "topk": wl.k,
            "max_visible_rows": spec.max_scored,
            "mean_visible_rows": float(np.mean([(int(p) + 1) // wl.ratio for p in wl.q_pos])),
            "attention_layers": wl.layers,
            "l2": "inputs larger than L2: the index plane read per step is "
                  f"{index_bytes / 1e6:.0f} MB",
            "parallelism": f"dp{world} (independent sequence batches per GPU)",
            "steps_per_graph": G,
        },
        "achieved_hbm_gbs": total_bytes / (ms_step / 1e3) / 1e9,
        "algorithmic_bytes_per_step": total_bytes,
        "roofline": {
            "kernel": "csa2_compress_index_topk stage (index prep + tcgen05 score kernel + "
                      "top-k, the compressor's tokens on extra top-k CTAs)",
            "bound": "hbm",
            "achieved": achieved_index,
            "peak": peak,
            "peak_kind": f"{peak_kind} hbm_gbs",
            "unit": "GB/s",
            "frac": achieved_index / peak,
            "traffic": traffic_from_profile(args.config),
            "stage_ms": idx_ms,
            "stage_samples": n_samples,
            "algorithmic_bytes_per_launch": index_bytes,
        },
        "gpu_launches": kernel_launches(spec, t) * args.steps,
        "clocks": clk,
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_queries)
    if world == 1 and args.config == "decode" and not args.no_extra:
        line["other_configs"] = other_configs()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def bf16_peaks():
    """Measured dense bf16 tensor peaks (burst, sustained) in TFLOP/s, else the fallback."""
    try:
        with open(PEAKS) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


def index_flops(wl):
    """Tensor FLOPs of the index scores: 2 * H * 128 per scored (row, query) pair, counting
    only the visible rows (FULL) or the candidate rows (REINDEX) each query scores."""
    nvis = np.array([(int(p) + 1) // wl.ratio for p in wl.q_pos], dtype=np.int64)
    scored = np.full_like(nvis, wl.ncb * 8) if wl.reindex else nvis
    return float(scored.sum()) * 2 * wl.H * 128


def attn_flops(wl):
    """Tensor FLOPs of one attention layer: S = Q K^T and O = P V over each query's window
    (min(p + 1, 128) rows) and its selected rows, 64 heads x 512 dims."""
    nvis = np.array([(int(p) + 1) // wl.ratio for p in wl.q_pos], dtype=np.int64)
    scored = np.full_like(nvis, wl.ncb * 8) if wl.reindex else nvis
    rows = np.minimum(scored, wl.k) + np.minimum(np.asarray(wl.q_pos) + 1, 128)
    return float(rows.sum()) * 2 * 2 * 64 * 512


def other_configs():
    """The REINDEX, prefill and long configurations, each timed on this GPU: the device
    time of csa2_compress_index_topk (the index stage), of each attention layer and of the
    whole step (CUDA graphs of several calls, CUDA events), with the index stage's HBM
    fraction (decode-shaped configurations) or tensor fractions (prefill)."""
    import csa2_compressed_sparse_gb300 as csa2
    from csa2_compressed_sparse_gb300.step import allocate, run_step, swa_of
    peak_hbm, hbm_kind = hbm_peak()
    tf_burst, tf_sus, tf_kind = bf16_peaks()
    res = {}
    for name, inner, reps in (("reindex", 10, 20), ("long", 4, 10), ("prefill", 1, 4)):
        wl = make_workload(name, 0)
        spec = spec_for(wl)
        t = wl.materialize("cuda")
        buf = allocate(spec, t)
        run_step(spec, t, buf)
        torch.cuda.synchronize()
        csa2.csa2_device_status()
        cand = t.get("cand")

        def index_call():
            csa2.csa2_compress_index_topk(
                t["kv"], t["score"], t["cu_seqlens"], t["start_pos"], t["kv_state"],
                t["score_state"], t["plane"], t["inv_freq"], t["iq"], t["w"], t["index_k"],
                t["row_base"], t["q_seq"], t["q_pos"], spec.ratio, spec.k, spec.max_scored,
                buf.sel, buf.ws, sel_scores=buf.sel_scores, cand=cand, relu=spec.relu,
                eps=spec.eps)

        def attn_call(layer):
            fn = csa2.csa2_sparse_attn if layer == 0 else csa2.csa2_reuse_attn
            return lambda: fn(t["q"][layer], t["q_seq"], t["q_pos"], swa_of(spec, t, layer),
                              t["plane"], t["row_base"], buf.sel, t["sink"], buf.out[layer],
                              scale=spec.scale, ws=buf.attn_ws)

        idx_us = graph_time_us(index_call, inner, reps)
        att_us = [graph_time_us(attn_call(layer), inner, reps) for layer in range(wl.layers)]
        step_us = graph_time_us(lambda: run_step(spec, t, buf), inner, reps)
        csa2.csa2_device_status()
        total, index_b, attn_b = algorithmic_bytes(wl)
        index_b += total - index_b - attn_b * wl.layers  # the compressor's bytes
        r = {"workload": wl.name, "description": wl.description, "queries": wl.Q,
             "attention_layers": wl.layers,
             "stages_us": {"compress_index_topk": round(idx_us, 2),
                           "attention_per_layer": [round(x, 2) for x in att_us],
                           "step": round(step_us, 2)},
             "queries_per_s": wl.Q / (step_us * 1e-6)}
        if name == "prefill":
            fi, fa = index_flops(wl), attn_flops(wl)
            att_mean = sum(att_us) / len(att_us)
            r["index_tflops"] = fi / (idx_us * 1e-6) / 1e12
            r["attn_tflops"] = fa / (att_mean * 1e-6) / 1e12
            r["index_frac_of_bf16"] = {"burst": r["index_tflops"] / tf_burst,
                                       "sustained": r["index_tflops"] / tf_sus}
            r["attn_frac_of_bf16"] = {"burst": r["attn_tflops"] / tf_burst,
                                      "sustained": r["attn_tflops"] / tf_sus}
            r["formula"] = ("tflops = tensor FLOPs / device time; index FLOPs = 2 H 128 per "
                            "scored (row, query); attention FLOPs = 2 x 2 x 64 x 512 per "
                            "(row, query), rows = window + selected; peaks: " + tf_kind +
                            f" bf16 {tf_burst:.0f} (burst) / {tf_sus:.0f} (sustained) TFLOP/s")
        else:
            r["index_gbs"] = index_b / (idx_us * 1e-6) / 1e9
            r["index_hbm_frac"] = r["index_gbs"] / peak_hbm
            r["step_gbs"] = total / (step_us * 1e-6) / 1e9
            r["step_hbm_frac"] = r["step_gbs"] / peak_hbm
            r["formula"] = ("GB/s = algorithmic bytes / device time (index: 256 B per scored "
                            "row + queries, weights, selection, candidate ids, compressor "
                            "tokens; step: every stage's bytes); peak: " + hbm_kind +
                            f" copy {peak_hbm:.0f} GB/s")
        res[name] = r
        del t, buf
        torch.cuda.empty_cache()
    return res


def run_e2e(args, wl, spec, t, buf, world, ms_step):
    """Each step copies its inputs from pinned host memory, runs the step through the
    C ABI and reads the outputs back; timed on the host and on the stream.

    The step's small inputs (new tokens, queries, positions, weights) live in one
    contiguous device buffer per slot and are filled by one copy from one pinned host
    buffer; the outputs (attention output of every layer, the selection) likewise leave
    in one copy.  Two slots alternate, so the copies of one step run on their own
    streams while the neighbouring step computes; the steps themselves stay in order on
    one compute stream (they share the planes and the workspace), each a CUDA graph of
    the same C-ABI calls."""
    import csa2_compressed_sparse_gb300 as csa2
    from csa2_compressed_sparse_gb300.step import run_step
    names = ["kv", "score", "iq", "w", "q_pos", "q_seq", "cu_seqlens", "start_pos"]
    align = 256

    def layout(tensors):
        offs, o = [], 0
        for x in tensors:
            offs.append(o)
            o += (x.numel() * x.element_size() + align - 1) // align * align
        return offs, max(o, align)

    def views(flat, tensors, offs):
        return [flat[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape)
                for x, o in zip(tensors, offs)]

    ins = [t[n] for n in names] + list(t["q"])
    outs = list(buf.out) + [buf.sel]
    in_offs, in_bytes = layout(ins)
    out_offs, out_bytes = layout(outs)
    h2d = sum(x.numel() * x.element_size() for x in ins)
    d2h = sum(x.numel() * x.element_size() for x in outs)
    slots = []
    for _ in range(2):
        d_in = torch.empty(in_bytes, dtype=torch.uint8, device="cuda")
        d_out = torch.empty(out_bytes, dtype=torch.uint8, device="cuda")
        h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        h_out = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
        for v, x in zip(views(h_in, ins, in_offs), ins):
            v.copy_(x.cpu())
        iv, ov = views(d_in, ins, in_offs), views(d_out, outs, out_offs)
        ts = dict(t)
        ts.update({n: v for n, v in zip(names, iv)})
        ts["q"] = iv[len(names):]
        bs = copy.copy(buf)
        bs.out, bs.sel = ov[:-1], ov[-1]
        slots.append((d_in, d_out, h_in, h_out, ts, bs))
    comp, cp_in, cp_out, side = (torch.cuda.Stream() for _ in range(4))
    graphs = []
    for d_in, d_out, h_in, h_out, ts, bs in slots:
        d_in.copy_(h_in)
        comp.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(comp):
            run_step(spec, ts, bs, side=side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=comp):
            run_step(spec, ts, bs, side=side)
        graphs.append(g)
    torch.cuda.synchronize()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}
    # at least half a second of steps, whatever --steps is
    steps = max(20, args.steps // 10, int(0.5e3 / max(ms_step, 1e-3)) + 1)

    def run(n):
        for i in range(n):
            s = i & 1
            d_in, d_out, h_in, h_out, _, _ = slots[s]
            if i >= 2:
                cp_in.wait_event(ev["comp"][s])   # step i-2 has read this slot's inputs
            with torch.cuda.stream(cp_in):
                d_in.copy_(h_in, non_blocking=True)
                ev["in"][s].record(cp_in)
            comp.wait_event(ev["in"][s])
            if i >= 2:
                comp.wait_event(ev["out"][s])     # step i-2's outputs have left
            with torch.cuda.stream(comp):
                graphs[s].replay()
                ev["comp"][s].record(comp)
            cp_out.wait_event(ev["comp"][s])
            with torch.cuda.stream(cp_out):
                h_out.copy_(d_out, non_blocking=True)
                ev["out"][s].record(cp_out)

    run(4)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    e0.record(cp_in)
    run(steps)
    cp_out.wait_stream(comp)
    e1.record(cp_out)
    torch.cuda.synchronize()
    wall = max_over_ranks(time.perf_counter() - w0, world, "cuda")
    csa2.csa2_device_status()
    return {"value": weak_value(wl.Q, world, steps, wall * 1e3), "unit": "queries/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "device_ms_per_step": e0.elapsed_time(e1) / steps, "steps": steps,
            "copies": "one packed H2D and one packed D2H per step, overlapped with the "
                      "neighbouring step's compute (two slots)"}


# ---- CPU oracle legs ------------------------------------------------------------------------

def oracle_step(wl, queries):
    """The oracle on a subset of queries: compress their sequences' new tokens, index,
    top-k, and every attention layer.  Returns seconds of oracle work."""
    import oracle
    import synth
    from oracle.harness import HostSeq, query_inputs, window_rows
    prep = []
    for q in queries:
        b = int(wl.q_seq[q])
        iq, w = query_inputs(wl, q)
        k_rows = synth.rows_bf16(b, 0, int(wl.n_rows[b]), 128, wl.seed, synth.INDEX_K)
        prep.append((q, b, iq, w, k_rows))
    t0 = time.perf_counter()
    sels = {}
    seqs = {}
    for q, b, iq, w, k_rows in prep:
        if b not in seqs:
            seqs[b] = HostSeq(wl, b)   # the oracle compressor over the step's tokens
        cand = None if wl.cand is None else wl.cand[q:q + 1]
        sc, rows = oracle.index_scores(iq, w, k_rows, [0], [0], [int(wl.q_pos[q])], wl.ratio,
                                       cand=cand)
        sels[q] = oracle.topk(sc[0], rows[0], wl.k)
    t_index = time.perf_counter() - t0
    # attention: one batched oracle call per layer over the sampled queries
    t_attn = 0.0
    for layer in range(wl.layers):
        qs, planes, sel_c, wins = [], [], [], []
        base = 0
        for q, b, *_ in prep:
            s = sels[q]
            v = s >= 0
            planes.append(seqs[b].plane_rows(s[v]))
            sc = np.full(len(s), -1, dtype=np.int32)
            sc[v] = base + np.arange(int(v.sum()))
            base += int(v.sum())
            sel_c.append(sc)
            qs.append(wl.host_q(q, layer))
            wins.append(window_rows(wl, q, layer))
        plane = oracle.bf16_from_bits(np.concatenate(planes)) if base else torch.zeros((1, 512), dtype=torch.bfloat16)
        sink = synth.normal_f32(64, wl.seed, synth.SINK)
        t1 = time.perf_counter()
        for i, (q, b, *_) in enumerate(prep):
            w = wins[i]
            oracle.sparse_attn(qs[i].view(1, 64, 512), [0], [int(wl.q_pos[q])], w["swa"], plane,
                               [0], sel_c[i].reshape(1, -1), sink, swa_mode=w["swa_mode"],
                               lin_base=w["lin_base"], lin_pos0=w["lin_pos0"])
        t_attn += time.perf_counter() - t1
    return t_index + t_attn


def cpu_baseline(wl, nq):
    import oracle  # noqa: F401  (built on first use)
    qs = list(range(min(nq, wl.Q)))
    secs = oracle_step(wl, qs)
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {"value": len(qs) / secs, "unit": "queries/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(qs)} of {wl.Q} queries of one step ({wl.name}): oracle compressor, "
                      f"indexer, top-k and {wl.layers} attention layer(s); {secs:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    wl = make_workload(args.config, 0)
    nq = min(8, wl.Q)
    qs = list(range(nq))
    for _ in range(args.warmup):
        oracle_step(wl, qs[:1])
    tot = 0.0
    for i in range(args.steps):
        tot += oracle_step(wl, qs)
    value = nq * args.steps / tot
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "queries/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "description": wl.description,
                   "sample_queries_per_step": nq},
        "cpu_baseline": {"value": value, "unit": "queries/s", "cores": cores, "kind": "oracle",
                         "sample": f"{nq} queries of {wl.name} per step"},
        "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def graph_time_us(fn, inner=20, reps=20):
    """Mean device time (us) of one fn() call: `inner` calls captured in one CUDA graph,
    replayed `reps` times between CUDA events on the launching stream (3 untimed replays
    first)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(inner):
            fn()
    for _ in range(3):
        g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (inner * reps)


def run_stages(args):
    """Mean device time of each entry point on the chosen workload: 20 calls captured in
    one CUDA graph, replayed `reps` times between CUDA events on the launching stream."""
    import csa2_compressed_sparse_gb300 as csa2
    from csa2_compressed_sparse_gb300.step import allocate, run_step, swa_of
    torch.cuda.set_device(0)
    wl = make_workload(args.config, 0)
    spec = spec_for(wl)
    t = wl.materialize("cuda")
    buf = allocate(spec, t)
    for _ in range(3):
        run_step(spec, t, buf)
    torch.cuda.synchronize()
    csa2.csa2_device_status()

    timed = graph_time_us

    cand = t.get("cand")
    swa0 = swa_of(spec, t, 0)
    res = {}
    res["compress"] = timed(lambda: csa2.csa2_compress(
        t["kv"], t["score"], t["cu_seqlens"], t["start_pos"], spec.ratio, t["kv_state"],
        t["score_state"], t["plane"], t["row_base"], t["inv_freq"], eps=spec.eps))
    # index K produced inside the compressor (wk, k_norm, RoPE): seeded weights of the pages' shapes
    g = np.random.default_rng(5)
    wk = torch.from_numpy((g.standard_normal((128, 512)) / np.sqrt(512)).astype(np.float32))
    wk = wk.bfloat16().cuda()
    kw = torch.ones(128, dtype=torch.float32, device="cuda")
    iplane = torch.empty((t["plane"].shape[0], 128), dtype=torch.bfloat16, device="cuda")
    res["compress_index"] = timed(lambda: csa2.csa2_compress_index(
        t["kv"], t["score"], t["cu_seqlens"], t["start_pos"], spec.ratio, t["kv_state"],
        t["score_state"], t["plane"], t["row_base"], t["inv_freq"], wk, iplane, knorm_w=kw,
        eps=spec.eps))
    res["index_topk"] = timed(lambda: csa2.csa2_index_topk(
        t["iq"], t["w"], t["index_k"], t["row_base"], t["q_seq"], t["q_pos"], spec.ratio, spec.k,
        spec.max_scored, buf.sel, buf.ws, sel_scores=buf.sel_scores, cand=cand))
    if cand is None:
        nbk = 2048
        pws = torch.empty(csa2.csa2_index_topk_pool_workspace_size(
            wl.Q, spec.H, spec.max_scored, spec.k, nbk), dtype=torch.uint8, device="cuda")
        pool = torch.empty((wl.Q, nbk), dtype=torch.int32, device="cuda")
        res["index_topk_pool"] = timed(lambda: csa2.csa2_index_topk_pool(
            t["iq"], t["w"], t["index_k"], t["row_base"], t["q_seq"], t["q_pos"], spec.ratio,
            spec.k, spec.max_scored, buf.sel, pool, pws, sel_scores=buf.sel_scores))
    # the FP8 index plane: sequences re-laid on 8-row blocks, quantised once
    from csa2_compressed_sparse_gb300.step import fp8_index_plane
    plane8, rb8, rows8 = fp8_index_plane(t["index_k"], wl.row_base, wl.n_rows)
    ws8 = torch.empty(csa2.csa2_index_topk_fp8_workspace_size(wl.Q, spec.H, spec.max_scored,
                                                               spec.k),
                      dtype=torch.uint8, device="cuda")
    sel8 = torch.empty_like(buf.sel)
    res["index_topk_fp8"] = timed(lambda: csa2.csa2_index_topk_fp8(
        t["iq"], t["w"], plane8, rows8, rb8, t["q_seq"], t["q_pos"], spec.ratio, spec.k,
        spec.max_scored, sel8, ws8, cand=cand))
    # the MXFP4 index plane: the same re-laying, quantised once
    from csa2_compressed_sparse_gb300.step import block_index_plane
    plane4i, rb4, rows4 = block_index_plane(t["index_k"], wl.row_base, wl.n_rows, "fp4")
    ws4 = torch.empty(csa2.csa2_index_topk_fp4_workspace_size(wl.Q, spec.H, spec.max_scored,
                                                               spec.k),
                      dtype=torch.uint8, device="cuda")
    sel4 = torch.empty_like(buf.sel)
    res["index_topk_fp4"] = timed(lambda: csa2.csa2_index_topk_fp4(
        t["iq"], t["w"], plane4i, rows4, rb4, t["q_seq"], t["q_pos"], spec.ratio, spec.k,
        spec.max_scored, sel4, ws4, cand=cand))
    res["sparse_attn"] = timed(lambda: csa2.csa2_sparse_attn(
        t["q"][0], t["q_seq"], t["q_pos"], swa0, t["plane"], t["row_base"], buf.sel, t["sink"],
        buf.out[0], scale=spec.scale, ws=buf.attn_ws))
    res["sparse_attn_rope"] = timed(lambda: csa2.csa2_sparse_attn_rope(
        t["q"][0], t["q_seq"], t["q_pos"], swa0, t["plane"], t["row_base"], buf.sel, t["sink"],
        buf.out[0], t["inv_freq"], scale=spec.scale, ws=buf.attn_ws))
    # the FP4 main plane: the same rows quantised once
    rows = t["plane"].shape[0]
    p4 = torch.empty(csa2.csa2_plane_fp4_bytes(rows), dtype=torch.uint8, device="cuda")
    csa2.csa2_plane_fp4(t["plane"], p4)
    res["sparse_attn_fp4"] = timed(lambda: csa2.csa2_sparse_attn_fp4(
        t["q"][0], t["q_seq"], t["q_pos"], swa0, p4, rows, t["row_base"], buf.sel, t["sink"],
        buf.out[0], scale=spec.scale, ws=buf.attn_ws))
    res["step"] = timed(lambda: run_step(spec, t, buf))
    csa2.csa2_device_status()
    print(json.dumps({"stages_us": {k: round(v, 2) for k, v in res.items()},
                      "workload": wl.name, "description": wl.description,
                      "queries": wl.Q}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.stages:
        run_stages(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
