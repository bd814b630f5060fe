#!/usr/bin/env python3
"""Decode-step benchmark of the low-bit KV cache on GB300.

One step = for every layer: append one new token per sequence
(kv_quant_append, which flushes the fp16 window into packed groups when it
fills) and attend one query token per (sequence, query head) over the whole
cache (kv_decode_attn).  Inputs (new K/V tokens, queries) and the cache are
resident in HBM; the cache of all layers together is far larger than L2, so
every layer's read comes from HBM.

Metric: decode-attention context tokens/s/layer = sum over sequences of the
tokens attended, divided by the time of one layer (step time / layers).  The
JSON line also carries the roofline of the decode-attention call (algorithmic
bytes / CUDA-event time against the measured HBM copy bandwidth), timed
before the steps on the workload's own state (context + 1 tokens per
sequence), the prefill's quantize kernel, the CPU
oracle's throughput on a bounded sample, and an end-to-end number through the
same C ABI with host buffers copied in and out every step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (times the CPU oracle instead)
"""

import os

# the CPU oracle runs single-threaded so its core count is exact
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import dataclasses  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import re  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_kv_cache_02_gb300 import synth  # noqa: E402

METRIC = "decode-attn context tokens/s/layer & achieved HBM GB/s vs 8 TB/s"  # value: the tokens/s; roofline: the GB/s
UNIT = "context tokens/s/layer"
DEFAULT_WORKLOAD = "llama2_7b_mha"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    p.add_argument("--layers", type=int, default=0, help="override the workload's layer count")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-oracle sample")
    p.add_argument("--warps", type=int, default=0, help="warps a decode launch cuts its work into (0: library's choice)")
    p.add_argument("--no-configs", action="store_true", help="skip the decode/quantize roofline of the other workloads")
    return p.parse_args()


# --------------------------------------------------------------------- setup

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world, device):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0}, "fallback"


def decode_bytes(lengths, w):
    """Algorithmic HBM bytes of one layer's decode attention: every packed
    group block (K/V codes + fp32 metadata) once, every fp16 sink/window
    token (K and V) once, the query and the output."""
    from bit_kv_cache_02_gb300.kvq import block_bytes
    bb = block_bytes(w.bits, key_per_token=w.key_per_token, outliers=w.dense_sparse)
    total = 0
    for L in lengths:
        ns = min(L, w.num_sink)
        n = L - ns
        r = n % w.residual
        total += w.kv_heads * ((n - r) // 32 * bb + (r + ns) * 2 * 128 * 2)
    total += len(lengths) * w.q_heads * 128 * 2 * 2
    return total


def kernel_source_hash(names=("decode_kernel.cuh", "kvq_internal.cuh")):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "bit_kv_cache_02_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


QUANT_SOURCES = ("quant.cu", "quant_tiles.cu", "quant_common.cuh", "kvq_internal.cuh")


def ncu_traffic(profile, algorithmic_bytes, sources=("decode_kernel.cuh", "kvq_internal.cuh")):
    """DRAM bytes per call: the committed ncu summary's ratio of captured DRAM
    traffic to the captured launch's algorithmic bytes, scaled to this run's
    algorithmic bytes per call; None unless the summary was taken on the
    current kernel source."""
    path = os.path.join(ROOT, "profiles", profile)
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_per_algorithmic_byte:\s*([0-9.]+)\s+source_hash:\s*([0-9a-f]+)", text)
    if not m or m.group(2) != kernel_source_hash(sources):
        return None
    return float(m.group(1)) * algorithmic_bytes


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        self.gpu = ids[local_rank] if local_rank < len(ids) else str(local_rank)
        self.proc = None
        self.file = None
        self.window = None

    def mark(self, t0, t1):
        """Wall-clock bounds of the timed region (samples outside are dropped)."""
        self.window = (t0, t1)

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        import datetime
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                if self.window and not (self.window[0] - 0.05 <= ts <= self.window[1] + 0.05):
                    continue
                rows.append(parts[1:])
        os.unlink(self.file.name)
        sm = [float(r[1]) for r in rows if _num(r[1])]
        mx = [float(r[2]) for r in rows if _num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _json_default(o):
    if hasattr(o, "item"):
        return o.item()
    raise TypeError(f"not JSON serializable: {type(o).__name__}")


def _num(s):
    try:
        float(s)
        return True
    except ValueError:
        return False


# ---------------------------------------------------------- our arm (GPU)

def prefill_lengths(w, untimed):
    """Prefilled tokens per sequence: the workload's context lengths plus its
    new token, less the untimed steps appended before the timed regions, so
    that decode attention is timed on the workload's own state (L = context
    + 1 per sequence: 4096 quantized tokens and a one-token window for the
    Llama-2 shape); the timed steps continue from there."""
    base = synth.context_lengths(w)
    return np.maximum(base + 1 - untimed, 1).astype(np.int64)


def prefill_bytes(lengths, w):
    """Algorithmic bytes of a prefill: quantized tokens read fp16 K and V and
    write their share of the packed blocks; window and sink tokens are read
    and written as fp16."""
    from bit_kv_cache_02_gb300.kvq import block_bytes
    bb = block_bytes(w.bits, key_per_token=w.key_per_token, outliers=w.dense_sparse)
    total = 0
    for L in lengths:
        L = int(L)
        ns = min(L, w.num_sink)
        n = L - ns
        r = n % w.residual
        total += w.kv_heads * ((n - r) * (2 * 128 * 2 + bb // 32) + (r + ns) * 2 * 2 * 128 * 2)
    return total


def build_caches(kvq, w, layers, pre, capacity, device):
    """Prefill every layer's cache (kv_quant_append of the whole context);
    returns the caches and the per-layer prefill times (CUDA events).  The
    call's host cost is kept out of the timed interval: a short device-side
    wait is queued before the start event, so the call's kernels are already
    queued behind it when the start event fires (otherwise the GPU sits idle
    between the event and the first kernel while the host marshals and
    checks the call's arguments)."""
    caches, times = [], []
    stream = torch.cuda.current_stream(device)
    for layer in range(layers):
        c = kvq.KVCache(w.seqs, w.kv_heads, capacity, bits=w.bits, residual=w.residual, num_sink=w.num_sink,
                        pre_rope=w.pre_rope, device=device, key_per_token=w.key_per_token,
                        paged=w.paged, hadamard=w.hadamard, outliers=w.dense_sparse)
        if w.paged:
            tbl = synth.block_table(w, layer, w.seqs, w.kv_heads, c.max_groups)
            c.block_table.copy_(torch.from_numpy(tbl).to(device))
        T = int(pre.max())
        k, v = synth.kv_tokens(w, layer, T, device=device)
        k, v = k.contiguous(), v.contiguous()
        nl = torch.as_tensor(pre.astype(np.int32), device=device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(2_000_000)  # about 1 ms of device time ahead of the start event
        e0.record(stream)
        kvq.kv_quant_append(c, k, v, nl, T, stream=stream)
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3)
        del k, v
        caches.append(c)
    torch.cuda.synchronize()
    for c in caches:
        if int(c.status.item()) != 0:
            raise RuntimeError(f"prefill reported device status {int(c.status.item())}")
    return caches, times


def run_ours(args, w, layers, rank, world, local):
    from bit_kv_cache_02_gb300 import build
    build.build()
    from bit_kv_cache_02_gb300 import kvq

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.warps:
        kvq.set_decode_warps(args.warps)
    K, W = args.steps, args.warmup
    pool = max(1, min(4, K))
    pre = prefill_lengths(w, max(W, 1) + pool)
    capacity = int(pre.max()) + max(W, 1) + pool + K + 64   # room for the end-to-end steps too
    caches, prefill_s = build_caches(kvq, w, layers, pre, capacity, device)
    prefill = {"seconds_per_layer": statistics.median(prefill_s), "bytes_per_layer": prefill_bytes(pre, w),
               "seconds_min_max": (min(prefill_s), max(prefill_s))}

    S, Hq = w.seqs, w.q_heads
    k_new = [[synth.kv_tokens(w, l, 1, device=device, stream_id=1 + p) for l in range(layers)] for p in range(pool)]
    qs = [[synth.queries(w, l, p, device=device) for l in range(layers)] for p in range(pool)]
    ones = torch.ones(S, dtype=torch.int32, device=device)
    outs = [torch.empty((S, Hq, 128), dtype=torch.float16, device=device) for _ in range(layers)]
    # The decode grid is sized for the cache capacity, so one captured graph
    # serves every step (the kernel reads the actual lengths on the device).
    max_len = capacity
    ws = kvq.alloc_workspace(caches[0], Hq, max_len)  # zero-filled; every layer's call leaves it so

    def step_calls(p, append=True):
        for l in range(layers):
            if append:
                kn, vn = k_new[p][l]
                kvq.kv_quant_append(caches[l], kn, vn, ones, 1)
            kvq.kv_decode_attn(caches[l], qs[p][l], outs[l], ws, max_len)

    # eager warm-up, then one CUDA graph per input set: a step launches ~3
    # kernels per layer, too many to issue from Python at the GPU's pace
    for i in range(max(W, 1)):
        step_calls(i % pool)
    torch.cuda.synchronize()
    n0 = kvq.launch_count()
    graphs = []
    for p in range(pool):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step_calls(p)
        graphs.append(g)
    launches_per_step = (kvq.launch_count() - n0) // pool
    dgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dgraph):
        step_calls(0, append=False)
    for p in range(pool):                 # first replays upload the graphs
        graphs[p].replay()
    torch.cuda.synchronize()
    done = max(W, 1) + pool                # steps appended so far
    attn_lens = pre + done                 # the workload's state: context + 1 per sequence
    lens_at = [attn_lens + 1 + i for i in range(K)]   # lengths attended in timed step i
    stream = torch.cuda.current_stream(device)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    wall_d0 = time.time()
    # decode attention alone, on the workload's state: the same calls
    # without the appends, replayed (the state does not change)
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    dgraph.replay()
    torch.cuda.synchronize()
    d0.record(stream)
    for _ in range(K):
        dgraph.replay()
    d1.record(stream)
    torch.cuda.synchronize()
    attn_avg_s = d0.elapsed_time(d1) / 1e3 / (K * layers)

    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t0.record(stream)
    for i in range(K):
        graphs[i % pool].replay()
    t1.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(wall_d0, time.time())   # both timed regions
    barrier(world)
    clocks = sampler.stop() if sampler else None
    elapsed_ms = t0.elapsed_time(t1)
    final_lens = attn_lens + K
    for c in caches:
        if int(c.status.item()) != 0:
            raise RuntimeError(f"device status {int(c.status.item())} after the timed steps")

    tokens_per_layer_step = [int(l.sum()) for l in lens_at]
    local_tokens = float(sum(tokens_per_layer_step)) * layers      # context tokens attended, all layers
    elapsed_ms = max_over_ranks(elapsed_ms, world, device)
    total_tokens = sum_over_ranks(local_tokens, world, device)
    # tokens/s/layer = (tokens one layer attends) / (step time / layers)
    value = total_tokens / (elapsed_ms / 1e3)
    bytes_avg = decode_bytes(attn_lens, w)
    attn_tokens_per_s = float(attn_lens.sum()) / attn_avg_s

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(kvq, w, caches, layers, k_new, qs, ones, outs, ws, max_len, final_lens, world, device)

    return dict(value=value, elapsed_ms=elapsed_ms, attn_avg_s=attn_avg_s, bytes_avg=bytes_avg,
                attn_tokens_per_s=attn_tokens_per_s, clocks=clocks, launches=launches_per_step * K,
                mean_ctx=float(np.mean([l.mean() for l in lens_at])), attn_ctx=float(attn_lens.mean()),
                e2e=e2e, prefill=prefill,
                cache_bytes=sum(c.blocks.numel() + 4 * c.k_res.numel() for c in caches))


def run_e2e(kvq, w, caches, layers, k_new, qs, ones, outs, ws, max_len, lens0, world, device):
    """The same steps through the same C ABI, with every step's inputs (new K/V
    token and query of every layer) copied from pinned host memory and every
    output copied back to pinned host memory inside the timed region, and the
    host waiting for each step's outputs before the next.  A step's inputs
    arrive together: they are staged in one pinned host buffer per kind and
    copied in one transfer each; the per-layer calls take views of the
    device copies, and all layers' outputs go back in one transfer.  As a
    serving loop would, the step's calls are captured once in a CUDA graph
    and replayed: the graph holds the copies in, every layer's
    kv_quant_append and kv_decode_attn and the copy out, so every replay
    moves that step's bytes.  The same steps issued eagerly from Python are
    timed too (eager_value).  The caches continue from their current state
    (one more token per step)."""
    pool = len(k_new)
    h_kv = [torch.stack([torch.stack([k_new[p][l][j] for l in range(layers)]) for j in range(2)]).cpu().pin_memory()
            for p in range(pool)]                                   # [2][layers][S][Hkv][1][D]
    h_q = [torch.stack([qs[p][l] for l in range(layers)]).cpu().pin_memory() for p in range(pool)]
    d_kv = torch.empty(h_kv[0].shape, dtype=h_kv[0].dtype, device=device)
    d_q = torch.empty(h_q[0].shape, dtype=h_q[0].dtype, device=device)
    d_out = torch.empty((layers,) + tuple(outs[0].shape), dtype=outs[0].dtype, device=device)
    h_out = torch.empty(d_out.shape, dtype=d_out.dtype).pin_memory()
    h2d = (d_kv.numel() + d_q.numel()) * 2
    d2h = d_out.numel() * 2

    def step_calls(p):
        d_kv.copy_(h_kv[p], non_blocking=True)
        d_q.copy_(h_q[p], non_blocking=True)
        for l in range(layers):
            kvq.kv_quant_append(caches[l], d_kv[0, l], d_kv[1, l], ones, 1)
            kvq.kv_decode_attn(caches[l], d_q[l], d_out[l], ws, max_len)
        h_out.copy_(d_out, non_blocking=True)

    def timed(run_step, n, state):
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(n):
            run_step(i % pool)
            torch.cuda.synchronize()  # the step's outputs are in host memory
        elapsed = max_over_ranks(time.perf_counter() - t0, world, device)
        tokens = sum_over_ranks(float(sum(int((state + 1 + i).sum()) for i in range(n))) * layers, world, device)
        return tokens / elapsed

    state = lens0.copy()
    n_eager = 10
    eager = timed(step_calls, n_eager, state)
    state = state + n_eager
    graphs = []
    for p in range(pool):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step_calls(p)
        graphs.append(g)
    for g in graphs:   # first replays upload the graphs (one step each)
        g.replay()
    torch.cuda.synchronize()
    state = state + pool
    n_steps = 20
    value = timed(lambda p: graphs[p].replay(), n_steps, state)
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n_steps, "eager_value": eager, "eager_steps": n_eager,
            "timer": "host perf_counter around each step's graph replay (pinned host -> device copies, "
                     "append + decode of every layer, device -> pinned host copies) and a synchronize",
            "eager_timer": "host perf_counter around the same calls issued eagerly from Python, per step "
                           "synchronized"}


# ------------------------------------------------- the other workloads

CONFIG_WORKLOADS = ("tiny", "llama3_8b_gqa_2bit", "llama3_8b_gqa_4bit", "long_1m", "kvquant_prerope")


def run_config(kvq, name, device, replays, peak):
    """One workload besides the headline one, timed as the headline is:
    caches prefilled to the workload's own state (context + its decode
    tokens), the prefill's kv_quant_append timed per layer with CUDA events,
    then K replays of a CUDA graph of kv_decode_attn over the layers.  Two
    layers (each cache larger than L2, so the pair of them is far larger)
    for multi-layer workloads; the one-layer workloads as they are (the
    million-token cache is 3.25 GiB; Tiny is launch-bound)."""
    w = synth.WORKLOADS[name]
    layers = min(w.layers, 2)
    state = synth.context_lengths(w).astype(np.int64) + w.decode_tokens
    capacity = int(state.max()) + 8
    caches, prefill_s = build_caches(kvq, w, layers, state, capacity, device)
    qs = [synth.queries(w, l, 0, device=device) for l in range(layers)]
    outs = [torch.empty_like(q) for q in qs]
    ws = kvq.alloc_workspace(caches[0], w.q_heads, capacity)
    for l in range(layers):
        kvq.kv_decode_attn(caches[l], qs[l], outs[l], ws, capacity)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for l in range(layers):
            kvq.kv_decode_attn(caches[l], qs[l], outs[l], ws, capacity)
    g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(replays):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    for c in caches:
        if int(c.status.item()) != 0:
            raise RuntimeError(f"{name}: device status {int(c.status.item())}")
    call_s = e0.elapsed_time(e1) / 1e3 / (replays * layers)
    dbytes = decode_bytes(state, w)
    qbytes = prefill_bytes(state, w)
    q_s = statistics.median(prefill_s)
    out = {"state_tokens_mean": float(state.mean()), "layers_timed": layers, "replays": replays,
           "decode_us": call_s * 1e6, "algorithmic_bytes": dbytes, "achieved_gbs": dbytes / call_s / 1e9,
           "frac": dbytes / call_s / 1e9 / peak, "traffic": ncu_traffic(f"decode_attn_{name}.md", dbytes), "context_tokens_per_s_per_layer": float(state.sum()) / call_s,
           "quantize_us": q_s * 1e6, "quantize_bytes": qbytes, "quantize_frac": qbytes / q_s / 1e9 / peak}
    del caches, qs, outs, ws, g
    torch.cuda.empty_cache()
    return out


def run_configs(args, device, peak):
    from bit_kv_cache_02_gb300 import build
    build.build()
    from bit_kv_cache_02_gb300 import kvq
    res = {}
    for name in CONFIG_WORKLOADS:
        if name == args.workload:
            continue
        try:
            res[name] = run_config(kvq, name, device, max(args.steps, 10), peak)
        except Exception as e:  # one workload's failure is reported, not fatal
            res[name] = {"unavailable": f"{type(e).__name__}: {e}"}
    return res


# ------------------------------------------------------------ CPU oracle

class OracleSample:
    """The CPU oracle on a bounded sample of the workload: n (sequence, KV
    head) pairs of layer 0 prefilled (untimed) to the workload's mean
    context; each step appends one token per pair and runs the oracle's
    attention for all query heads of those KV heads.  The step time is
    scaled linearly from n pairs to the whole layer (S x Hkv pairs)."""

    def __init__(self, w, seconds_per_step):
        import oracle
        self.w = w
        self.ctx = int(synth.context_lengths(w).mean())
        self.gq = w.q_heads // w.kv_heads
        self.pairs = w.seqs * w.kv_heads
        probe = self._make(oracle, 1, 4)
        t = time.perf_counter()
        self._step(probe, 0)
        per_pair = max(time.perf_counter() - t, 1e-4)
        self.n = int(max(1, min(self.pairs, seconds_per_step / per_pair)))
        self.state = self._make(oracle, self.n, 256)
        self.i = 0

    def _make(self, oracle, n, extra):
        ws = dataclasses.replace(self.w, seqs=n, kv_heads=1, q_heads=self.gq, ragged_min=0, ctx=self.ctx)
        k, v = synth.kv_tokens(ws, 0, self.ctx + extra)
        k, v = k.numpy(), v.numpy()
        c = oracle.OracleCache(n, 1, self.ctx + extra, self.w.bits, residual=self.w.residual,
                               num_sink=self.w.num_sink, key_per_token=self.w.key_per_token,
                               hadamard=self.w.hadamard, outliers=self.w.dense_sparse)
        c.append(k[:, :, :self.ctx], v[:, :, :self.ctx], [self.ctx] * n)
        return ws, k, v, c

    def _step(self, state, i):
        ws, k, v, c = state
        j = self.ctx + i
        c.append(k[:, :, j:j + 1], v[:, :, j:j + 1], [1] * c.S)
        c.attention(synth.queries(ws, 0, i).numpy(), pre_rope=self.w.pre_rope)
        return int(c.seq_len.mean())

    def step(self):
        """One timed step: (context tokens of the whole layer, scaled seconds)."""
        t = time.perf_counter()
        L = self._step(self.state, self.i % 250)
        dt = time.perf_counter() - t
        self.i += 1
        return L * self.w.seqs, dt * self.pairs / self.n

    def describe(self, steps):
        return (f"{self.n} of {self.pairs} (sequence, KV head) pairs of layer 0 at context {self.ctx}, "
                f"{steps} steps of append + attention ({self.gq} query heads per KV head), "
                f"step time scaled linearly to all pairs")


def oracle_throughput(w, budget_s):
    """(tokens/s/layer, description) of the oracle over about budget_s."""
    smp = OracleSample(w, budget_s / 8)
    tok = sec = 0.0
    steps = 0
    t0 = time.perf_counter()
    while steps < 8 and (steps == 0 or time.perf_counter() - t0 < budget_s):
        a, b = smp.step()
        tok, sec, steps = tok + a, sec + b, steps + 1
    return tok / sec, smp.describe(steps)


def cpu_cores_used():
    return 1


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def host_cpu_model():
    """The host CPU's model name: lscpu's, else /proc/cpuinfo's (Arm cores
    report an implementer and a part number there instead of a name)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    arm_parts = {"0xd0c": "Neoverse N1", "0xd40": "Neoverse V1", "0xd49": "Neoverse N2", "0xd4f": "Neoverse V2",
                 "0xd8e": "Neoverse N3", "0xd84": "Neoverse V3"}
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "cpu part" in fields:
        return arm_parts.get(fields["cpu part"], f"Arm core, part {fields['cpu part']}")
    import platform
    return platform.processor() or platform.machine()


def _oracle_worker(name, per_step, steps, barrier, results):
    """One process of the all-cores oracle run: its own bounded sample (built
    untimed), then `steps` timed steps started together with the others."""
    w = synth.WORKLOADS[name]
    smp = OracleSample(w, per_step)
    smp.step()                                    # warm-up
    barrier.wait(timeout=180)
    t0 = time.perf_counter()
    for _ in range(steps):
        smp.step()
    results.put((smp.n, steps, time.perf_counter() - t0))


def oracle_throughput_all_cores(w, per_step=1.0, steps=3):
    """The same oracle on every host core at once: one process per core, each
    stepping its own sample of (sequence, KV head) pairs; the aggregate
    pair-steps per second over the slowest process's time, scaled to the
    layer's context tokens.  Processes are spawned (no fork of this one)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    n_proc = host_cores()
    barrier = ctx.Barrier(n_proc)
    results = ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(w.name, per_step, steps, barrier, results))
             for _ in range(n_proc)]
    for p in procs:
        p.start()
    import queue
    got = []
    deadline = time.time() + 240
    try:
        while len(got) < n_proc:
            try:
                got.append(results.get(timeout=5))
            except queue.Empty:
                failed = [p.exitcode for p in procs if p.exitcode not in (None, 0)]
                if failed or time.time() > deadline:
                    raise RuntimeError(f"oracle processes failed (exit codes {failed}) or ran out of time")
    finally:
        for p in procs:   # only the processes started here
            p.join(timeout=10)
            if p.is_alive():
                p.terminate()
    pair_steps = sum(n * k for n, k, _ in got)
    wall = max(t for _, _, t in got)
    pairs = w.seqs * w.kv_heads
    ctx_tokens = int(synth.context_lengths(w).mean())
    value = pair_steps / wall / pairs * ctx_tokens * w.seqs
    desc = (f"{n_proc} processes, each {got[0][0]} (sequence, KV head) pairs of layer 0 at context "
            f"{ctx_tokens}, {steps} steps of append + attention, timed together; pair-steps per second "
            f"scaled to the whole layer")
    return value, n_proc, desc


# ------------------------------------------------------------------- main

def main():
    args = parse_args()
    rank, world, local = dist_env()
    w = synth.WORKLOADS[args.workload]
    layers = args.layers or w.layers
    config = {"workload": w.name, "layers": layers, "seqs_per_gpu": w.seqs, "q_heads": w.q_heads,
              "kv_heads": w.kv_heads, "head_dim": 128, "ctx": w.ctx, "bits": w.bits, "group": 32,
              "residual": w.residual, "num_sink": w.num_sink, "pre_rope": w.pre_rope,
              "key_per_token": w.key_per_token,
              "paged": w.paged,
              "hadamard": w.hadamard,
              "outliers": w.dense_sparse,
              "ragged": bool(w.ragged_min), "parallelism": f"replicas{world}",
              "l2": "inputs larger than L2: each layer's packed cache is streamed once per step"}

    if args.impl == "reference":
        init_dist(world, "gloo")
        if rank != 0:
            barrier(world)
            return
        per_step = min(2.0, 150.0 / max(1, args.steps + args.warmup))
        smp = OracleSample(w, per_step)
        for _ in range(args.warmup):
            smp.step()
        t0 = time.perf_counter()
        tok = sec = 0.0
        for _ in range(args.steps):
            a, b = smp.step()
            tok, sec = tok + a, sec + b
        total = time.perf_counter() - t0
        value = tok / sec
        desc = smp.describe(args.steps)
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores_used(), "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line, default=_json_default))
        barrier(world)
        return

    init_dist(world, "nccl")
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc = oracle_throughput(w, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cpu_cores_used(), "kind": "oracle", "sample": desc,
               "cpu_model": host_cpu_model()}
        try:
            va, na, desca = oracle_throughput_all_cores(w)
            cpu["all_cores"] = {"value": va, "unit": UNIT, "cores": na, "kind": "oracle", "sample": desca}
        except Exception as e:  # the single-core figure stands on its own
            cpu["all_cores"] = {"unavailable": f"{type(e).__name__}: {e}"}
    r = run_ours(args, w, layers, rank, world, local)
    peaks, which = measured_peaks()
    configs = None
    if not args.no_configs:
        torch.cuda.empty_cache()
        configs = run_configs(args, torch.device("cuda", local), float(peaks["hbm_gbs"]))
    if rank != 0:
        return
    achieved = r["bytes_avg"] / r["attn_avg_s"] / 1e9
    peak = float(peaks["hbm_gbs"])
    traffic = ncu_traffic(f"decode_attn_{w.name}.md", r["bytes_avg"])
    q_traffic = ncu_traffic(f"quant_prefill_{w.name}.md", r["prefill"]["bytes_per_layer"], QUANT_SOURCES)
    line = {
        "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["elapsed_ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": f"u{w.bits}-codes/f32-accum",
        "data": "synthetic", "config": dict(config, mean_ctx_timed=r["mean_ctx"], attn_ctx=r["attn_ctx"]),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "frac_of_nominal_8tbs": achieved / 8000.0, "traffic": traffic,
                     "kernel": "decode_kernel (one per kv_decode_attn call)", "peak_source": which,
                     "timing": "CUDA events around K replays of a graph of 32 kv_decode_attn calls",
                     "algorithmic_bytes_per_call": r["bytes_avg"], "call_us": r["attn_avg_s"] * 1e6},
        "attn_only": {"value": r["attn_tokens_per_s"], "unit": UNIT},
        "quantize": {"kernel": "kv_quant_append (prefill of one layer)",
                     "achieved": r["prefill"]["bytes_per_layer"] / r["prefill"]["seconds_per_layer"] / 1e9,
                     "unit": "GB/s", "peak": peak,
                     "frac": r["prefill"]["bytes_per_layer"] / r["prefill"]["seconds_per_layer"] / 1e9 / peak,
                     "algorithmic_bytes": r["prefill"]["bytes_per_layer"], "traffic": q_traffic,
                     "us": r["prefill"]["seconds_per_layer"] * 1e6,
                     "us_min_max_over_layers": [round(x * 1e6, 1) for x in r["prefill"]["seconds_min_max"]]},
        "configs": configs,
        "cpu_baseline": cpu,
        "e2e": r["e2e"],
        "gpu_launches": r["launches"],
        "timing": "CUDA events around K replays of CUDA graphs, one graph per decode step",
        "clocks": r["clocks"],
    }
    print(json.dumps(line, default=_json_default))


if __name__ == "__main__":
    main()
