"""Benchmark of the paged-KV attention hot path on GB300.

One step = one decode step of a Qwen3-0.6B-shaped model at c=64 over its 28
attention layers: for every layer, the KV store of the 64 new tokens (one per
sequence, position 639) into that layer's paged cache, then paged decode
attention of the 64 sequences at context 640 (16 query heads, 8 KV heads,
head_dim 128, block size 256). Every layer has its own seeded cache (168 MB of
K/V per layer, 4.7 GB per step, far larger than the 129 MB L2), so nothing is
reused from L2 between layers or steps. The headline value is seq*layer/s.

The same JSON line also carries:
  roofline      the decode call (split + merge kernels) as the dominant kernel:
                algorithmic bytes per call / average call duration in the
                graph-timed region (CUDA events around it / calls in it),
                against the measured HBM copy bandwidth; the eager loop's
                per-call event time beside it;
  prefill       the prefix-cached prefill (8 x 4096 new tokens over a shared
                4096-token cached prefix, 1.649 TFLOP per call) in TFLOP/s,
                against the measured bf16 tensor peak; and the KV store of
                those 32768 tokens in GB/s;
  e2e           the same step through the Python API with host (pinned) inputs
                and outputs, copies inside the timed region;
  cpu_baseline  the fp64 oracle on the host cores, on a bounded sample.

`--impl reference` times the oracle alone (the reference arm).
Under torchrun, every rank runs its own replica of the workload (its own
sequences; weak scaling) and the time is the maximum over ranks.
"""
import argparse
import ctypes
import hashlib
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

import workloads as W  # noqa: E402

METRIC = ("paged decode attn HBM GB/s (% of peak) & seq·layer/s; "
          "prefill attn TFLOP/s")
LAYERS = W.NUM_LAYERS
DECODE_SEQS = 64
DECODE_CTX = 640


# ---------------------------------------------------------------- arithmetic

def decode_algorithmic_bytes(num_seqs, ctx, H_q=W.H_Q, H_kv=W.H_KV, D=W.HEAD_DIM, bs=256,
                             window=0):
    """Bytes a decode call must move at least: K and V rows of the attended
    tokens (the last `window` with a sliding window), q, out, lse, the used
    block-table entries and the context length."""
    first = ctx - window if 0 < window < ctx else 0
    kv = (ctx - first) * H_kv * D * 2 * 2
    q_out = 2 * H_q * D * 2
    lse = H_q * 4
    table = (-(-ctx // bs) - first // bs) * 4
    return num_seqs * (kv + q_out + lse + table + 4)


def kv_store_algorithmic_bytes(num_tokens, H_kv=W.H_KV, D=W.HEAD_DIM):
    """Read k and v rows, write them into the cache, read the slot."""
    return num_tokens * (H_kv * D * 2 * 2 * 2 + 4)


def prefill_flops(q_lens, k_lens, H_q=W.H_Q, D=W.HEAD_DIM, window=0):
    """4*D FLOPs per unmasked (query, key, head): Q K^T and P V. Query i of a
    segment sees Lk - Lq + i + 1 keys, at most `window` with a sliding window."""
    pairs = 0
    for lq, lk in zip(q_lens, k_lens):
        lq, lk = int(lq), int(lk)
        if window <= 0:
            pairs += lq * (lk - lq) + lq * (lq + 1) // 2
        else:
            n = np.arange(lk - lq + 1, lk + 1, dtype=np.int64)  # keys of each query
            pairs += int(np.minimum(n, window).sum())
    return 4 * D * pairs * H_q


def weight_streaming_roof(bandwidth_bytes_s, weight_bytes, concurrency):
    """Crude decode roof of a model that streams its weights once per step:
    tokens/s = bandwidth / weight bytes x concurrency."""
    return bandwidth_bytes_s / weight_bytes * concurrency


# ---------------------------------------------------------------- environment

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                source="fallback")


def source_digest(*names):
    h = hashlib.sha1()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_attention_22_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def profiled_traffic(kernel, digest):
    """DRAM bytes per launch from the committed ncu summary of `kernel`, if it
    was taken from the current source (same digest); else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_digest") != digest:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        self.result = None
        if self.proc is None:
            return False
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if sm:
            self.result = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                           "reasons": sorted(reasons), "samples": len(sm)}
        return False


# ---------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(backend):
    rank, world, local = dist_env()
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)
    return rank, world, local


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def max_over_ranks(x: float, device=None) -> float:
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, device=None) -> float:
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- GPU legs

def _dev(a):
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class Sweep:
    """The layers' device state and pre-marshalled C-ABI calls."""

    def __init__(self, pkv, seed_base, num_layers=LAYERS, window=0, shard_world=1):
        """window: sliding window of every decode call (0: none). shard_world > 1:
        the caches, q and new rows of one rank's KV-head shard only (tensor
        parallelism over that many ranks; every rank's shard is the same work)."""
        from paged_kv_attention_22_gb300.shard import head_shard, take_heads
        self.pkv = pkv
        self.L = pkv.lib()
        self.window = int(window)
        self.layers = []
        self.host_cases = []
        for layer in range(num_layers):
            case = W.sweep64_layer(layer, base_seed=seed_base)
            qh, kvh = head_shard(0, shard_world, case.H_q, case.H_kv)
            hk = lambda a: take_heads(a, kvh, 1)
            pool = take_heads(case.poisoned_pool(), kvh, 2)
            kc, vc = _dev(pool), _dev(pool)
            pkv.kv_store(_dev(hk(case.history.k)), _dev(hk(case.history.v)), kc, vc,
                         _dev(case.history.slots))
            st = case.step
            q = take_heads(st.q, qh, 1)
            S, H_q, D = q.shape
            H_kv = pool.shape[2]
            d = dict(kc=kc, vc=vc, q=_dev(q), k=_dev(hk(st.new.k)), v=_dev(hk(st.new.v)),
                     slots=_dev(st.new.slots), bt=_dev(case.block_tables),
                     ctx=_dev(st.context_lens), out=torch.empty((S, H_q, D), dtype=torch.bfloat16,
                                                                 device="cuda"),
                     lse=torch.empty((S, H_q), dtype=torch.float32, device="cuda"))
            d["ws"] = pkv.new_decode_workspace(S, H_q, H_kv, D, st.max_context_len)
            self.layers.append(d)
            self.host_cases.append(case)
        torch.cuda.synchronize()
        if pkv.check_device_errors() != 0:
            raise RuntimeError("device error while filling the caches")
        c0 = self.host_cases[0]
        self.S, self.H_q, self.D = self.layers[0]["q"].shape
        self.H_kv = self.layers[0]["kc"].shape[2]
        self.bs, self.NB = c0.block_size, c0.num_blocks
        self.max_ctx = c0.step.max_context_len
        self.scale = c0.scale

    def calls(self, stream_handle, fused=True):
        """Per layer, the C-ABI calls of one decode step as (function, args) pairs:
        the fused store+decode call, or the KV store then the decode."""
        P = ctypes.c_void_p
        L = self.L
        out = []
        for d in self.layers:
            common = (P(d["q"].data_ptr()), P(d["kc"].data_ptr()), P(d["vc"].data_ptr()),
                      P(d["bt"].data_ptr()), d["bt"].shape[1], P(d["ctx"].data_ptr()),
                      self.max_ctx, self.S, self.H_q, self.H_kv, self.D, self.bs, self.NB,
                      ctypes.c_float(self.scale), self.window, P(d["out"].data_ptr()),
                      P(d["lse"].data_ptr()),
                      P(d["ws"].data_ptr()), d["ws"].numel(), P(stream_handle))
            if fused:
                # the caches, tables and lengths of a decode step are set before
                # it: each call may read them while the previous one finishes
                out.append([(L.pkv_paged_decode_attn_store,
                             (P(d["k"].data_ptr()), P(d["v"].data_ptr()),
                              P(d["slots"].data_ptr())) + common[:-1] +
                             (self.pkv.DECODE_STABLE_INPUTS, common[-1]))])
            else:
                out.append([(L.pkv_kv_store,
                             (P(d["k"].data_ptr()), P(d["v"].data_ptr()), P(d["kc"].data_ptr()),
                              P(d["vc"].data_ptr()), P(d["slots"].data_ptr()), d["k"].shape[0],
                              self.H_kv, self.D, self.bs, self.NB, P(stream_handle))),
                            (L.pkv_paged_decode_attn, common)])
        return out

    def run_step(self, calls, events=None):
        """Issue one step; with events, bracket each layer's last (decode) call."""
        L = self.L
        for i, layer in enumerate(calls):
            for j, (fn, args) in enumerate(layer):
                last = j == len(layer) - 1
                if events is not None and last:
                    events[i][0].record()
                if fn(*args) != 0:
                    raise RuntimeError("pkv call failed: " + L.pkv_last_cuda_error().decode())
                if events is not None and last:
                    events[i][1].record()


def time_sweep(sweep, steps, warmup, device, fused=True):
    stream = torch.cuda.current_stream()
    calls = sweep.calls(stream.cuda_stream, fused)
    for _ in range(warmup):
        sweep.run_step(calls)
    torch.cuda.synchronize()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(len(sweep.layers))] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    start.record()
    for k in range(steps):
        sweep.run_step(calls, ev[k])
    end.record()
    torch.cuda.synchronize()
    barrier()
    total_ms = start.elapsed_time(end)
    decode_ms = [a.elapsed_time(b) for row in ev for a, b in row]
    return total_ms, decode_ms


def time_sweep_graph(sweep, steps, warmup, fused=True):
    """The same step captured once into a CUDA graph and replayed."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        calls = sweep.calls(s.cuda_stream, fused)
        sweep.run_step(calls)  # warm the stream before capture
        s.synchronize()
        with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
            sweep.run_step(sweep.calls(s.cuda_stream, fused))
    torch.cuda.synchronize()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        g.replay()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def _packed(tensors, device):
    """One byte buffer holding the given tensors back to back (256-byte aligned
    parts), and views of it shaped like them."""
    offs, off = [], 0
    for t in tensors:
        offs.append(off)
        off += -(-(t.numel() * t.element_size()) // 256) * 256
    buf = torch.empty(off, dtype=torch.uint8, device=device)
    if device == "cpu":
        buf = buf.pin_memory()
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
             for o, t in zip(offs, tensors)]
    return buf, views


def time_e2e(sweep, steps, warmup):
    """Through the Python API with pinned host buffers: per step, one copy of
    every layer's q, new k, new v and slots from a packed pinned host buffer to
    the device, the 28 fused calls on views of it, and one copy of every
    layer's out and lse back to a packed pinned host buffer. The copies run on
    their own streams into and out of two alternating device buffers, so step
    k+1's inputs move while step k computes; events order every buffer's use."""
    pkv = sweep.pkv
    names = ("q", "k", "v", "slots")
    ins = [sweep.layers[i][k] for i in range(len(sweep.layers)) for k in names]
    outs = [t for d in sweep.layers for t in (d["out"], d["lse"])]
    host_in, host_views = _packed(ins, "cpu")
    for hv, t in zip(host_views, ins):
        hv.copy_(t.cpu())
    dev_in = [_packed(ins, "cuda") for _ in range(2)]
    dev_out = [_packed(outs, "cuda") for _ in range(2)]
    host_out = [_packed(outs, "cpu")[0] for _ in range(2)]
    nk = len(names)
    h2d = host_in.numel()
    d2h = host_out[0].numel()
    compute = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready, in_free = [ev(), ev()], [ev(), ev()]
    out_ready, out_free = [ev(), ev()], [ev(), ev()]
    for b in range(2):  # both buffers start free
        in_free[b].record(compute)
        out_free[b].record(compute)

    def step(k):
        b = k & 1
        (din, in_views), (dout, out_views) = dev_in[b], dev_out[b]
        up.wait_event(in_free[b])                 # compute of step k-2 is done with it
        with torch.cuda.stream(up):
            din.copy_(host_in, non_blocking=True)
        in_ready[b].record(up)
        compute.wait_event(in_ready[b])
        compute.wait_event(out_free[b])           # step k-2's outputs have been copied out
        for i, d in enumerate(sweep.layers):
            q, kk, v, slots = in_views[nk * i:nk * (i + 1)]
            pkv.paged_decode_attn_store(kk, v, slots, q, d["kc"], d["vc"], d["bt"], d["ctx"],
                                        sweep.max_ctx, sweep.scale, out=out_views[2 * i],
                                        lse=out_views[2 * i + 1], workspace=d["ws"],
                                        stable_inputs=True)
        in_free[b].record(compute)
        out_ready[b].record(compute)
        down.wait_event(out_ready[b])
        with torch.cuda.stream(down):
            host_out[b].copy_(dout, non_blocking=True)
        out_free[b].record(down)

    for k in range(warmup):
        step(k)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(compute)
    up.wait_event(start)                          # the first copy in starts after `start`
    for k in range(steps):
        step(k)
    for b in range(2):
        compute.wait_event(out_free[b])           # every result is back on the host
    end.record(compute)
    torch.cuda.synchronize()
    return start.elapsed_time(end), h2d, d2h


def time_prefill(pkv, steps, warmup, window=0):
    """Prefix-cached prefill: store of the 32768 prompt tokens, then prefill;
    then the decode step at context 8193 on the same cache (both with the
    given sliding window)."""
    pre, dec = W.prefix8k()
    kc, vc = _dev(pre.poisoned_pool()), _dev(pre.poisoned_pool())
    pkv.kv_store(_dev(pre.history.k), _dev(pre.history.v), kc, vc, _dev(pre.history.slots))
    st = pre.step
    k, v, slots = _dev(st.new.k), _dev(st.new.v), _dev(st.new.slots)
    q, cq, ck, bt = _dev(st.q), _dev(st.cu_seqlens_q), _dev(st.cu_seqlens_k), _dev(pre.block_tables)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[0], q.shape[1]), dtype=torch.float32, device="cuda")
    # Each leg times n calls back to back between two events on the stream,
    # so that a call's host work (tensor maps, launch) overlaps the previous
    # call's kernels instead of adding to the device time.
    n = max(steps, 20)

    def prefill_call():
        pkv.paged_prefill_attn(q, kc, vc, cq, ck, bt, st.max_seqlen_q, st.max_seqlen_k, pre.scale,
                               out=out, lse=lse, sliding_window=window)

    def timed_run(call):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            call()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    pkv.kv_store(k, v, kc, vc, slots)
    for _ in range(max(warmup, 3)):
        prefill_call()
    torch.cuda.synchronize()
    pkv.kv_store(k, v, kc, vc, slots)  # the store runs first; the calls queue behind it
    pre_ms = timed_run(prefill_call)
    if pkv.check_device_errors() != 0:
        raise RuntimeError("device error in the prefill leg")
    store_ms = time_kv_store(pkv, k, v, slots, pre) if window == 0 else None
    flops = prefill_flops(np.diff(st.cu_seqlens_q), np.diff(st.cu_seqlens_k), window=window)
    store_bytes = kv_store_algorithmic_bytes(st.new.num_tokens)

    # decode of one token per sequence at context 8193 over the shared prefix
    ds = dec.step
    pkv.kv_store(_dev(ds.new.k), _dev(ds.new.v), kc, vc, _dev(ds.new.slots))
    dq, dlen = _dev(ds.q), _dev(ds.context_lens)
    dout = torch.empty_like(dq)
    dlse = torch.empty((dq.shape[0], dq.shape[1]), dtype=torch.float32, device="cuda")
    ws = pkv.new_decode_workspace(dq.shape[0], dq.shape[1], W.H_KV, W.HEAD_DIM,
                                  ds.max_context_len)
    def dec_call():
        pkv.paged_decode_attn(dq, kc, vc, bt, dlen, ds.max_context_len, dec.scale, out=dout,
                              lse=dlse, workspace=ws, sliding_window=window)

    for _ in range(max(warmup, 3)):
        dec_call()
    torch.cuda.synchronize()
    pkv.kv_store(k, v, kc, vc, slots)  # a kernel ahead of the first call, as above
    dec_ms = timed_run(dec_call)
    if pkv.check_device_errors() != 0:
        raise RuntimeError("device error in the prefix decode leg")
    ctx = int(ds.context_lens[0])
    S = int(ds.context_lens.shape[0])
    logical = decode_algorithmic_bytes(S, ctx, window=window)
    # the cached prefix every sequence attends (none of it inside a window that
    # ends 4097 tokens later)
    shared_tokens = 4096 if window <= 0 or window > ctx - 4096 else 0
    unique = logical - (S - 1) * shared_tokens * W.H_KV * W.HEAD_DIM * 2 * 2
    return dict(prefill_ms=pre_ms, flops=flops, store_ms=store_ms, store_bytes=store_bytes,
                decode_ms=dec_ms, decode_logical_bytes=logical,
                decode_unique_bytes=unique)


def time_kv_store(pkv, k, v, slots, case, pools=4, n_short=8, n_long=24):
    """Milliseconds per KV store of the prompt tokens, as the slope between
    n_short and n_long back-to-back stores: the stores rotate over `pools`
    destination cache pairs (pools x 160 MB, several times the 129 MB L2), so
    each store's cache lines are written back to DRAM while later stores run,
    and the dirty lines left in L2 when the timed region ends are the same for
    both counts and cancel in the difference."""
    dst = [(_dev(case.poisoned_pool()), _dev(case.poisoned_pool())) for _ in range(pools)]

    def run(n):
        for _ in range(pools):  # the same starting state for every count
            for kc, vc in dst:
                pkv.kv_store(k, v, kc, vc, slots)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(n):
            kc, vc = dst[i % pools]
            pkv.kv_store(k, v, kc, vc, slots)
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    t_short = statistics.median(run(n_short) for _ in range(3))
    t_long = statistics.median(run(n_long) for _ in range(3))
    del dst
    return (t_long - t_short) / (n_long - n_short)


def time_block_manager(pkv, steps=200, seqs=64, prompt=640, shared=512, bs=256):
    """Host cost of the block manager through the Python API: admitting `seqs`
    prompts of `prompt` tokens that share their first `shared` tokens, then per
    decode step one appended token per sequence, its slot and the block-table
    rows of the batch (what a scheduler asks for each step)."""
    rng = np.random.default_rng(5)
    max_blocks = -(-(prompt + steps) // bs)
    bm = pkv.BlockManager(seqs * max_blocks, bs)
    head = rng.integers(0, 50000, shared).astype(np.int32)
    prompts = [np.concatenate([head, rng.integers(0, 50000, prompt - shared).astype(np.int32)])
               for _ in range(seqs)]
    t0 = time.perf_counter()
    cached = [bm.add_sequence(s, prompts[s]) for s in range(seqs)]
    admit_s = time.perf_counter() - t0
    toks = rng.integers(0, 50000, (steps, seqs)).astype(np.int32)
    t0 = time.perf_counter()
    for k in range(steps):
        slots = np.empty(seqs, np.int32)
        for s in range(seqs):
            bm.append_token(s, int(toks[k, s]))
            slots[s] = bm.slots(s, prompt + k, 1)[0]
        bm.block_tables(range(seqs), max_blocks)
    step_s = (time.perf_counter() - t0) / steps
    return {"workload": f"{seqs} prompts of {prompt} tokens sharing {shared}, block size {bs}; "
                        f"then {steps} decode steps (append, slot, block-table rows)",
            "admit_us_per_prompt": admit_s / seqs * 1e6,
            "cached_tokens_per_prompt": float(np.mean(cached[1:])),
            "us_per_decode_step": step_s * 1e6,
            "blocks_in_use": seqs * max_blocks - bm.num_free_blocks,
            "path": "python API over the C ABI (pkv_blocks.h)"}


# ---------------------------------------------------------------- CPU (oracle) legs

def oracle_sample(seconds_target=12.0, layers=4, seed_base=4000):
    """The fp64 oracle on a bounded sample of the sweep: `layers` layers of the
    64-sequence decode step (store + attention), repeated until about
    seconds_target seconds of host work. Returns (seq*layer/s, threads, desc)."""
    import oracle
    cases = [W.sweep64_layer(l, base_seed=seed_base) for l in range(layers)]
    caches = []
    for c in cases:
        kc, vc = c.poisoned_pool(), c.poisoned_pool()
        oracle.kv_store(c.history.k, c.history.v, kc, vc, c.history.slots)
        caches.append((kc, vc))
    done, t0 = 0, time.perf_counter()
    while True:
        for c, (kc, vc) in zip(cases, caches):
            st = c.step
            oracle.kv_store(st.new.k, st.new.v, kc, vc, st.new.slots)
            oracle.decode(st.q, kc, vc, c.block_tables, st.context_lens, c.scale)
            done += 1
        el = time.perf_counter() - t0
        if el >= seconds_target:
            break
    seq_layers = done * DECODE_SEQS
    desc = (f"{done} layer-steps ({layers} distinct layers) of the c=64 ctx-640 decode sweep, "
            f"{seq_layers} seq*layer in {el:.1f} s")
    return seq_layers / el, oracle.num_threads(), desc


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    per_step = []
    cases = [W.sweep64_layer(0)]
    kc, vc = cases[0].poisoned_pool(), cases[0].poisoned_pool()
    c = cases[0]
    oracle.kv_store(c.history.k, c.history.v, kc, vc, c.history.slots)
    st = c.step

    def step():
        oracle.kv_store(st.new.k, st.new.v, kc, vc, st.new.slots)
        oracle.decode(st.q, kc, vc, c.block_tables, st.context_lens, c.scale)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        t1 = time.perf_counter()
        step()
        per_step.append(time.perf_counter() - t1)
    total = time.perf_counter() - t0
    value = args.steps * DECODE_SEQS / total
    sample = ("each step: layer 0 of the 28-layer c=64 ctx-640 decode sweep "
              "(KV store of 64 tokens + decode of 64 sequences), fp64 oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "seq·layer/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "decode sweep c=64 ctx=640, 28 layers, bs=256, 16q/8kv x 128",
                   "sample": "one layer per step"},
        "cpu_baseline": {"value": value, "unit": "seq·layer/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "seq·layer/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- main

def time_extras(pkv, args, peaks, layers):
    """The sliding-window (SWA-256) decode sweep and prefix prefill, one rank's
    decode sweep on a 2-way KV-head shard, and the host block manager."""
    steps = max(args.steps // 2, 10)
    out = {}
    window = 256
    sw = Sweep(pkv, seed_base=4000, num_layers=layers, window=window)
    g_ms = time_sweep_graph(sw, steps, args.warmup)
    units = steps * layers * DECODE_SEQS
    nbytes = (decode_algorithmic_bytes(DECODE_SEQS, DECODE_CTX, window=window) +
              kv_store_algorithmic_bytes(DECODE_SEQS))
    per_layer = g_ms / 1000.0 / (steps * layers)
    out["window_decode"] = {"workload": f"c=64 ctx-640 decode sweep, {layers} layers, sliding "
                                        f"window {window} (fused store + decode per layer, graph)",
                            "value": units / (g_ms / 1000.0), "unit": "seq·layer/s",
                            "us_per_layer": per_layer * 1e6,
                            "gbs": nbytes / per_layer / 1e9,
                            "frac": nbytes / per_layer / 1e9 / peaks["hbm_gbs"]}
    del sw
    sh = Sweep(pkv, seed_base=4000, num_layers=layers, shard_world=2)
    g_ms = time_sweep_graph(sh, steps, args.warmup)
    per_layer = g_ms / 1000.0 / (steps * layers)
    nbytes = (decode_algorithmic_bytes(DECODE_SEQS, DECODE_CTX, H_q=8, H_kv=4) +
              kv_store_algorithmic_bytes(DECODE_SEQS, H_kv=4))
    out["head_shard_decode"] = {"workload": f"one rank of a 2-way KV-head shard (8 q / 4 kv "
                                            f"heads) of the c=64 ctx-640 sweep, {layers} layers",
                                "value_per_rank": units / (g_ms / 1000.0), "unit": "seq·layer/s",
                                "us_per_layer": per_layer * 1e6,
                                "gbs": nbytes / per_layer / 1e9,
                                "frac": nbytes / per_layer / 1e9 / peaks["hbm_gbs"]}
    del sh
    torch.cuda.empty_cache()
    pr = time_prefill(pkv, min(args.steps, 10), args.warmup, window=window)
    tflops = pr["flops"] / (pr["prefill_ms"] / 1000.0) / 1e12
    out["window_prefill"] = {"workload": f"prefix8k prefill with sliding window {window}",
                             "value": tflops, "unit": "TFLOP/s", "ms_per_call": pr["prefill_ms"],
                             "flops_per_call": pr["flops"],
                             "frac": tflops / peaks["bf16_tflops"],
                             "decode_us_per_call": pr["decode_ms"] * 1000.0,
                             "decode_gbs": pr["decode_logical_bytes"] / (pr["decode_ms"] / 1e3) / 1e9}
    torch.cuda.empty_cache()
    out["block_manager"] = time_block_manager(pkv)
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the decode sweep (profiling the prefill leg alone)")
    ap.add_argument("--decode-ctas", type=int, default=0,
                    help="persistent decode CTAs (0: one per SM)")
    ap.add_argument("--decode-variant", type=int, default=0,
                    help="decode launch shape (warps per CTA x stages per warp)")
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="layers per step (28 for the real workload; fewer for profiling)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the sliding-window, head-shard and block-manager legs")
    ap.add_argument("--prefill-window", type=int, default=0,
                    help="sliding window of the prefill leg (0: none; the windowed kernel "
                         "alone, for profiling)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return reference_arm(args)

    import paged_kv_attention_22_gb300 as pkv
    from paged_kv_attention_22_gb300 import build as pkv_build

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dist_init("nccl")
    if rank == 0:
        pkv_build.build()
    barrier()
    pkv.lib()
    pkv.decode_set_config(args.decode_ctas, args.decode_variant)

    # CPU baseline before any heavy GPU work (rank 0, N=1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, desc = oracle_sample()
        cpu = {"value": v, "unit": "seq·layer/s", "cores": cores, "kind": "oracle",
               "sample": desc}

    peaks = load_peaks()
    layers = args.layers
    value_graph = value_eager = t_max = g_max = None
    unfused = None
    roofline = None
    e2e = None
    clocks_result = None
    launches_per_step = 0
    if not args.no_sweep:
        sweep = Sweep(pkv, seed_base=4000 + 1000 * rank, num_layers=layers)
        with ClockSampler(local) as clocks:
            total_ms, decode_ms = time_sweep(sweep, args.steps, args.warmup, local)
            graph_ms = time_sweep_graph(sweep, args.steps, args.warmup)
        clocks_result = clocks.result
        # the same step as two calls per layer (KV store, then decode)
        _, unfused_dec_ms = time_sweep(sweep, args.steps, args.warmup, local, fused=False)
        unfused_graph_ms = time_sweep_graph(sweep, args.steps, args.warmup, fused=False)
        if pkv.check_device_errors() != 0:
            raise RuntimeError("device error during the timed region")
        t_max = max_over_ranks(total_ms / 1000.0, device="cuda")
        g_max = max_over_ranks(graph_ms / 1000.0, device="cuda")
        units = sum_over_ranks(args.steps * layers * DECODE_SEQS, device="cuda")
        value_eager = units / t_max
        value_graph = units / g_max
        dec_bytes = (decode_algorithmic_bytes(DECODE_SEQS, DECODE_CTX) +
                     kv_store_algorithmic_bytes(DECODE_SEQS))
        # The graph-timed region holds nothing but the step's decode calls, back
        # to back on one stream, so its event time / calls is the average call
        # duration as the headline value sees it. The eager loop's per-call
        # events (kept beside it) stop each call from overlapping its neighbours.
        call_s = graph_ms / 1000.0 / (args.steps * layers)
        achieved = dec_bytes / call_s / 1e9
        eager_s = statistics.mean(decode_ms) / 1000.0
        digest = source_digest("decode.cu", "ptx.cuh")
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "traffic": profiled_traffic("decode_kernel", digest),
                    "kernel": "decode call: decode_kernel (fused KV store + split-K) + decode_merge_kernel",
                    "algorithmic_bytes_per_launch": dec_bytes,
                    "us_per_launch": call_s * 1e6,
                    "timing": "CUDA events around the graph-replayed timed region on its "
                              "stream / decode calls in it",
                    "eager_us_per_call": eager_s * 1e6,
                    "eager_frac": dec_bytes / eager_s / 1e9 / peaks["hbm_gbs"],
                    "peak_kind": f"HBM copy ({peaks['source']})",
                    "source_digest": digest}
        launches_per_step = layers * 2  # fused store+decode kernel and merge kernel
        unfused = {"value": units / max_over_ranks(unfused_graph_ms / 1000.0, device="cuda"),
                   "decode_us_per_call": statistics.mean(unfused_dec_ms) * 1000.0,
                   "launches_per_step": layers * 3}
        if not args.no_e2e:
            n_e2e = max(args.steps // 4, 10)
            e_ms, h2d, d2h = time_e2e(sweep, n_e2e, args.warmup)
            e_max = max_over_ranks(e_ms / 1000.0, device="cuda")
            e_units = sum_over_ranks(n_e2e * layers * DECODE_SEQS, device="cuda")
            e2e = {"value": e_units / e_max, "unit": "seq·layer/s", "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h,
                   "path": "python API; per step one copy of the packed inputs in, the 28 "
                           "fused calls, one copy of the packed outputs back (pinned host); "
                           "the copies overlap the neighbouring steps' compute"}
        del sweep
        torch.cuda.empty_cache()

    prefill = None
    if not args.no_prefill:
        pr = time_prefill(pkv, min(args.steps, 20), args.warmup, window=args.prefill_window)
        tflops = pr["flops"] / (pr["prefill_ms"] / 1000.0) / 1e12
        # the store is timed with the unwindowed leg only
        store_gbs = (pr["store_bytes"] / (pr["store_ms"] / 1000.0) / 1e9
                     if pr["store_ms"] is not None else None)
        window_note = (f", sliding window {args.prefill_window}" if args.prefill_window > 0
                       else "")
        prefill = {"workload": "prefix-cached prefill: 8 seqs x 4096 new tokens over a shared "
                               "4096-token cached prefix (Lk 8192), bs=256" + window_note,
                   "value": tflops, "unit": "TFLOP/s", "ms_per_call": pr["prefill_ms"],
                   "flops_per_call": pr["flops"],
                   "frac": tflops / peaks["bf16_tflops"], "peak": peaks["bf16_tflops"],
                   "peak_kind": f"bf16 dense burst ({peaks['source']})",
                   "kv_store_gbs": store_gbs,
                   "kv_store_frac": (store_gbs / peaks["hbm_gbs"]
                                     if store_gbs is not None else None),
                   "timing": "20 calls back to back between two CUDA events, per call",
                   "kv_store_tokens": 32768,
                   "kv_store_timing": "slope between 8 and 24 back-to-back stores rotating over "
                                      "4 destination caches (640 MB, well above L2), so the "
                                      "write-back of the stored rows falls inside the timed "
                                      "region"}
        dsec = pr["decode_ms"] / 1000.0
        prefill["decode_after_prefix"] = {
            "workload": "decode of 8 seqs at context 8193 sharing the 4096-token prefix",
            "timing": "20 calls back to back between two CUDA events, per call",
            "us_per_call": pr["decode_ms"] * 1000.0,
            "logical_gbs": pr["decode_logical_bytes"] / dsec / 1e9,
            "unique_gbs": pr["decode_unique_bytes"] / dsec / 1e9,
            "logical_bytes": pr["decode_logical_bytes"],
            "unique_bytes": pr["decode_unique_bytes"],
            "frac_unique": pr["decode_unique_bytes"] / dsec / 1e9 / peaks["hbm_gbs"]}

    extras = None
    if not args.no_extras and not args.no_sweep and not args.no_prefill:
        extras = time_extras(pkv, args, peaks, layers=8)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": value_graph,
            "unit": "seq·layer/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": 1000.0 * g_max / args.steps if g_max else None,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"decode sweep c=64: 64 seqs x ctx 640, {layers} distinct "
                                   "layer caches, bs=256, 16 q / 8 kv heads x 128, KV store of "
                                   "the new token + decode per layer (one fused call)",
                       "timing": "CUDA graph of one step, replayed",
                       "l2": f"inputs larger than L2 ({layers * 168.3 / 1000:.1f} GB of K/V per "
                             "step, 168 MB per layer)",
                       "decode": "persistent split-K, one CTA per SM",
                       "decode_ctas": args.decode_ctas, "decode_variant": args.decode_variant},
            "eager": ({"value": value_eager, "ms_per_step": 1000.0 * t_max / args.steps}
                      if t_max else None),
            "unfused": unfused,
            "roofline": roofline,
            "prefill": prefill,
            "extras": extras,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks_result,
        }
        print(json.dumps(line))
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
