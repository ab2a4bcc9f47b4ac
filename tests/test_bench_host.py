"""Host-side logic of bench.py, without a GPU: the counting rules, the
reduction over ranks (two gloo ranks on CPU), and the reference arm's JSON."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import bench
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_decode_bytes_per_seq_layer():
    # 640 keys x 8 KV heads x 128 x 2 B x (K and V) + q + out + lse + 3 table entries + length
    per_seq = 640 * 8 * 128 * 2 * 2 + 2 * 16 * 128 * 2 + 16 * 4 + 3 * 4 + 4
    assert per_seq == 2_629_712
    assert bench.decode_algorithmic_bytes(64, 640) == 64 * per_seq


def test_prefill_flops_prefix8k():
    pre, _ = W.prefix8k()
    st = pre.step
    f = bench.prefill_flops(np.diff(st.cu_seqlens_q), np.diff(st.cu_seqlens_k))
    # per seq and head: 4096 x 4096 cached-prefix pairs + 4096 * 4097 / 2 causal pairs
    assert f == 4 * 128 * 16 * 8 * (4096 * 4096 + 4096 * 4097 // 2)
    assert abs(f - 1.649e12) < 1e9


def test_roofline_formula_reproduces_the_pages_anchors():
    path = os.path.join(ROOT, "tests", "golden", "sansho_roofline_anchors.txt")
    rows, vals = [], {}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        a, b = line.split()
        if a[0].isdigit():
            rows.append((int(a), int(b)))
        else:
            vals[a] = float(b)
    for c, printed in rows:
        got = bench.weight_streaming_roof(vals["bandwidth_bytes_per_s"], vals["weight_bytes"], c)
        assert round(got) == printed


def _ranks(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.dist_init("gloo")
    mx = bench.max_over_ranks(1.0 + rank)
    sm = bench.sum_over_ranks(10.0 * (rank + 1))
    bench.barrier()
    out[rank] = (mx, sm)
    torch.distributed.destroy_process_group()


def test_reductions_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_ranks, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (2.0, 30.0)


def test_reference_arm_prints_one_json_line():
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", "2", "--warmup", "3"], capture_output=True, text=True,
                          timeout=600, cwd=ROOT)
    assert proc.returncode == 0, proc.stderr
    lines = [l for l in proc.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "seq·layer/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_windowed_byte_and_flop_counts():
    # a window covering the context changes nothing
    assert bench.decode_algorithmic_bytes(3, 640, window=640) == bench.decode_algorithmic_bytes(3, 640)
    assert bench.decode_algorithmic_bytes(3, 640, window=5000) == bench.decode_algorithmic_bytes(3, 640)
    # window 256 of 640 keys: 256 K/V rows, blocks 1 and 2 of the table
    per_seq = 256 * 8 * 128 * 2 * 2 + 2 * 16 * 128 * 2 + 16 * 4 + 2 * 4 + 4
    assert bench.decode_algorithmic_bytes(64, 640, window=256) == 64 * per_seq
    # prefill: brute force over (query, key) pairs of a small ragged batch
    q_lens, k_lens, window = [5, 0, 9], [12, 3, 9], 4
    pairs = 0
    for lq, lk in zip(q_lens, k_lens):
        for i in range(lq):
            last = lk - lq + i
            pairs += sum(1 for p in range(lk) if last - window < p <= last)
    assert bench.prefill_flops(q_lens, k_lens, window=window) == 4 * W.HEAD_DIM * W.H_Q * pairs
    assert bench.prefill_flops(q_lens, k_lens, window=100) == bench.prefill_flops(q_lens, k_lens)


def test_block_manager_leg_runs_on_the_host():
    import paged_kv_attention_22_gb300 as pkv
    from paged_kv_attention_22_gb300 import build as pkv_build
    pkv_build.build()
    r = bench.time_block_manager(pkv, steps=20, seqs=8)
    assert r["cached_tokens_per_prompt"] == 512      # the shared 512 tokens are two full blocks
    assert r["us_per_decode_step"] > 0 and r["admit_us_per_prompt"] > 0
    # 2 shared blocks + one own block per sequence (its last 128 prompt tokens and
    # the 20 appended ones fit in it)
    assert r["blocks_in_use"] == 2 + 8
