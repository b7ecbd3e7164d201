"""Host-side logic on the CPU: seeded input generation, bench accounting, and the multi-rank
bench logic (seeds per rank, max-over-ranks timing, aggregate throughput) as world_size-2 gloo
processes."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from speculative_verify_gdn_gb300 import inputs as I


def test_inputs_are_seeded_and_reproducible():
    w = I.custom(I.WORKLOADS[1], name="host_small", L=2, B=3, N=4, V=512)
    a = I.round_stream(w, 3, seed=7)
    b = I.round_stream(w, 3, seed=7)
    c = I.round_stream(w, 4, seed=7)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert not torch.equal(a[0], c[0])
    lg1, dr1, L1 = I.greedy_logits(w, 1, seed=7)
    lg2, dr2, L2 = I.greedy_logits(w, 1, seed=7)
    assert torch.equal(lg1, lg2) and torch.equal(dr1, dr2) and torch.equal(L1, L2)
    g = a[1]
    assert float(g.min()) > 0 and float(g.max()) < 1
    beta = a[2]
    assert float(beta.min()) > 0 and float(beta.max()) < 1


def test_tree_generator_shape_rules():
    w = I.custom(I.WORKLOADS[4], name="host_tree", B=6)
    par = I.random_tree(w, 0).numpy()
    for b in range(w.B):
        p = par[b]
        assert all(-1 <= p[v] < v for v in range(w.N))
        depth = np.zeros(w.N, int)
        for v in range(w.N):
            depth[v] = 1 if p[v] < 0 else depth[p[v]] + 1
        assert depth.max() == w.tree_depth
        kids = np.bincount(p + 1, minlength=w.N + 1)
        assert kids.max() <= w.tree_branch
    tok, lg, L = I.tree_tokens_and_logits(w, torch.from_numpy(par), 0)
    for b in range(w.B):
        for u in range(-1, w.N):
            sib = tok[b][torch.from_numpy(par[b] == u)]
            assert len(set(sib.tolist())) == len(sib)


def test_bench_byte_accounting():
    w = I.WORKLOADS[2]
    S = 32 * 128 * 128 * 4
    per = S + 8 * (2 * 8192 + 8 * 32 + 2 * 32 * 128 + 4 * 32 * 128 + 4 * 16 * 128) + 2 * 3 * 8192
    assert bench.bytes_verify(w) == 30 * 64 * per + 30 * 2 * 8192 * 4
    assert bench.bytes_rollback(w, [0] * 64) == 4 * 64
    one = bench.bytes_rollback(w, [3] + [0] * 63) - 4 * 64
    assert one == 30 * (2 * S + 3 * (4 * 32 * 128 + 4 * 16 * 128 + 4 * 32) + 2 * 3 * 8192 * 2)
    # the rows the accept loop reaches: n + 1 per sequence
    assert bench.bytes_accept(w, [8] * 64) == 64 * 9 * 151936 * 2 + 4 * 64 * 18
    assert bench.bytes_accept(w, [0] * 63 + [3]) == (63 + 4) * 151936 * 2 + 4 * 64 * 18
    assert bench.aggregate_tokens_per_s(2, 64, 8, 2.0) == 2 * 64 * 8 / 2e-3


def test_bench_byte_accounting_gates_and_attention():
    import dataclasses
    w = I.WORKLOADS[2]
    # per-key-channel gates: the gate bytes grow from 4·Hv to 4·Hv·d per position, nothing else
    gdk = I.custom(w, name=w.name, gate_dk=True)
    assert bench.bytes_verify(gdk) - bench.bytes_verify(w) == 30 * 64 * 8 * 4 * 32 * 127
    assert (bench.bytes_rollback(gdk, [2] + [0] * 63) - bench.bytes_rollback(w, [2] + [0] * 63)
            == 30 * 2 * 4 * 32 * 127)
    aw = I.ATTN_WORKLOADS["qwen36_attn_b64_n8"]
    one = dataclasses.replace(aw, B=1)
    assert bench.bytes_attn(aw, [4096] * 64) == 64 * bench.bytes_attn(one, [4096])
    # one more committed row: one more key and value row read per layer and kv head
    assert (bench.bytes_attn(one, [4097]) - bench.bytes_attn(one, [4096])
            == 2 * aw.D * 2 * aw.L * aw.Hkv)
    # the per-step reads at 4096 rows dominate: K and V of 4104 rows x 10 layers x 2 kv heads
    assert bench.bytes_attn(one, [4096]) > 2 * 4104 * 256 * 2 * 10 * 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    ws, r = bench.init_dist("gloo")
    # each rank draws its own sequences; the timing reduction takes the slowest rank
    seed = bench.rank_seed(5, r)
    w = I.custom(I.WORKLOADS[1], name="host_rank", L=1, B=2, N=4, V=256)
    qkv, _, _ = I.round_stream(w, 0, seed=seed)
    ms = 10.0 + r
    t = bench.reduce_max(ms)
    bench.barrier()
    q.put((r, ws, seed, float(qkv.sum()), t,
           bench.aggregate_tokens_per_s(ws, w.B, w.N, t)))
    dist.destroy_process_group()


def test_two_rank_gloo_bench_logic():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ws0, s0, x0, t0, v0), (r1, ws1, s1, x1, t1, v1) = res
    assert ws0 == ws1 == 2
    assert s0 != s1 and x0 != x1                 # distinct sequences per rank
    assert t0 == t1 == 11.0                      # max over ranks
    assert v0 == v1 == pytest.approx(2 * 2 * 4 / 11e-3)


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON line with the
    contract's keys, on the default workload's metric and unit."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                       timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e",
                "cpu_baseline"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"
