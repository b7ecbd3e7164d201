"""Per-key-channel gates (the tape layout g [B, T, Hv, Dk] of the GDN investigation §4): the
oracle's per-channel branch pinned to its scalar branch (equal gates on every channel), to the
replay rule (tape replay of all T steps reaches the verify recurrence's final state) and to a
closed form (a zero gate on channel j erases column j), then (GPU) the CUDA path against it."""
import numpy as np
import pytest
import torch

import oracle
from test_oracle_pins import rand_inputs


def per_channel(g, D):
    """[..., Hv] gates repeated on every key channel -> [..., Hv, D]."""
    return np.repeat(np.asarray(g)[..., None], D, axis=-1)


@pytest.mark.parametrize("T,Hk,Hv,D", [(4, 2, 4, 8), (6, 1, 2, 16), (3, 2, 2, 4)])
def test_equal_channel_gates_reduce_to_the_scalar_gate(T, Hk, Hv, D):
    rng = np.random.default_rng(T * 100 + D)
    dims, x = rand_inputs(rng, L=2, B=2, T=T, Hk=Hk, Hv=Hv, D=D)
    a = oracle.verify(dims, x["qkv"], x["conv_w"], x["conv_state"], x["g"], x["beta"], x["state"])
    gdk = per_channel(x["g"], D)
    b = oracle.verify(dims, x["qkv"], x["conv_w"], x["conv_state"], gdk, x["beta"], x["state"])
    for key in ("out", "tape_delta", "tape_k"):
        np.testing.assert_allclose(b[key], a[key], rtol=1e-12, atol=1e-14)
    n = rng.integers(0, T + 1, size=2).astype(np.int32)
    s1, c1, bad1 = oracle.rollback(dims, n, a["tape_delta"], a["tape_k"], x["g"], x["qkv"],
                                   x["state"], x["conv_state"])
    s2, c2, bad2 = oracle.rollback(dims, n, a["tape_delta"], a["tape_k"], gdk, x["qkv"],
                                   x["state"], x["conv_state"])
    assert bad1 == bad2 == 0
    np.testing.assert_allclose(s2, s1, rtol=1e-12, atol=1e-14)
    assert np.array_equal(c1, c2)


def test_replay_of_every_step_reaches_the_sequential_state():
    rng = np.random.default_rng(7)
    T, D = 5, 8
    dims, x = rand_inputs(rng, L=1, B=2, T=T, Hk=2, Hv=4, D=D)
    gdk = np.exp(-np.logaddexp(0.0, rng.standard_normal((1, 2, T, 4, D))))
    ref = oracle.verify(dims, x["qkv"], x["conv_w"], x["conv_state"], gdk, x["beta"], x["state"],
                        node_states=True)
    st, _, bad = oracle.rollback(dims, np.array([T, T], np.int32), ref["tape_delta"],
                                 ref["tape_k"], gdk, x["qkv"], x["state"], x["conv_state"])
    assert bad == 0
    np.testing.assert_allclose(st, ref["node_state"][:, :, T - 1], rtol=1e-12, atol=1e-14)


def test_zero_gate_erases_its_key_column():
    rng = np.random.default_rng(11)
    T, D, j0 = 3, 8, 5
    dims, x = rand_inputs(rng, L=1, B=1, T=T, Hk=1, Hv=2, D=D)
    gdk = np.exp(-np.logaddexp(0.0, rng.standard_normal((1, 1, T, 2, D))))
    gdk[0, 0, T - 1, :, j0] = 0.0
    ref = oracle.verify(dims, x["qkv"], x["conv_w"], x["conv_state"], gdk, x["beta"], x["state"])
    st, _, _ = oracle.rollback(dims, np.array([T], np.int32), ref["tape_delta"], ref["tape_k"],
                               gdk, x["qkv"], x["state"], x["conv_state"])
    for h in range(2):
        col = ref["tape_delta"][0, 0, T - 1, h] * ref["tape_k"][0, 0, T - 1, h // 2, j0]
        np.testing.assert_allclose(st[0, 0, h, :, j0], col, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------------------------ GPU parity
def gdk_workload(D, T, io=torch.float32, L=2, B=4, Hk=2, Hv=4, W=4):
    from speculative_verify_gdn_gb300 import inputs as I
    return I.custom(I.WORKLOADS[1], name="gdk_D%d_T%d_H%d_%d_W%d_%s" % (D, T, Hk, Hv, W, str(io)),
                    L=L, B=B, N=T, Hk=Hk, Hv=Hv, D=D, W=W, V=64, io_dtype=io, gate_dk=True)


def run_gdk_verify_rollback(w, seed, n):
    from parity_util import assert_close, f64, oracle_rollback, oracle_verify, to_dev
    from speculative_verify_gdn_gb300 import inputs as I
    from speculative_verify_gdn_gb300.round import SpecRound
    cw = I.model_weights(w, seed)
    st, cs = I.initial_state(w, seed)
    qkv, g, beta = I.round_stream(w, 0, seed)
    assert g.shape == (w.L, w.B, w.N, w.Hv, w.D)
    r = SpecRound(w)
    dq, dcw, dcs, dg, db, dst = to_dev(qkv, cw, cs, g, beta, st)
    r.verify(dq, dcw, dcs, dg, db, dst)
    r.check_status()
    ref = oracle_verify(w, qkv, cw, cs, g, beta, st)
    bf16 = w.io_dtype == torch.bfloat16
    assert_close(f64(r.out), ref["out"], "out", bf16=bf16)
    assert_close(f64(r.tape_delta), ref["tape_delta"], "tape_delta")
    assert_close(f64(r.tape_k), ref["tape_k"], "tape_k")
    assert torch.equal(dst.cpu(), st)
    r.n_acc.copy_(torch.from_numpy(np.asarray(n, np.int32)))
    r.rollback(dq, dg, dst, dcs)
    r.check_status()
    st_ref, cs_ref, bad = oracle_rollback(w, n, ref, g, qkv, st, cs)
    assert bad == 0
    assert_close(f64(dst), st_ref, "state")
    assert np.array_equal(f64(dcs), cs_ref)


@pytest.mark.gpu
@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("T", [1, 4, 7, 16, 32])
def test_gpu_per_channel_gates_verify_and_rollback(gdnlib, D, T):
    w = gdk_workload(D, T)
    n = np.minimum(np.array([T, 0, 1, T // 2], np.int32), T)
    run_gdk_verify_rollback(w, T * 3 + D, n)


@pytest.mark.gpu
@pytest.mark.parametrize("Hk,Hv,T,W", [(2, 4, 8, 4), (4, 4, 16, 4), (1, 2, 5, 2), (2, 2, 8, 1)])
def test_gpu_per_channel_gates_bf16_qwen_heads(gdnlib, Hk, Hv, T, W):
    """bf16 I/O at d = 128 with one and two value heads per key head (the Qwen3.6 head shape)."""
    w = gdk_workload(128, T, io=torch.bfloat16, Hk=Hk, Hv=Hv, W=W)
    run_gdk_verify_rollback(w, Hk * 10 + Hv + T, np.array([T, 2, 0, T - 1], np.int32))


@pytest.mark.gpu
@pytest.mark.parametrize("Hk,Hv,T,W", [(2, 4, 1, 4), (2, 4, 3, 3), (1, 1, 4, 4), (2, 4, 4, 4),
                                       (3, 3, 7, 4), (2, 4, 6, 2)])
def test_gpu_per_channel_gates_pipelined_chain_lengths(gdnlib, Hk, Hv, T, W):
    """The pipelined kernel's per-key-channel path (bf16, d = 128, chains of T <= 8: one B tile
    per value head, the decayed Gram from the epilogue warps) at every chain-length class and
    both head groupings, then the rollback from its tape."""
    w = gdk_workload(128, T, io=torch.bfloat16, Hk=Hk, Hv=Hv, W=W, B=3)
    run_gdk_verify_rollback(w, 50 + T * 7 + Hv, np.array([T, 0, max(T - 1, 0)], np.int32))


@pytest.mark.gpu
def test_gpu_per_channel_gates_zero_gates_stay_exact(gdnlib):
    """Exact zero gates on some channels and positions (a closed key channel) on the pipelined
    path: the running-product Gram has no ratio of cumulative products, so nothing divides by
    the zero and the outputs match the oracle's per-step recurrence."""
    from parity_util import assert_close, f64, oracle_verify, to_dev
    from speculative_verify_gdn_gb300 import inputs as I
    from speculative_verify_gdn_gb300.round import SpecRound
    w = gdk_workload(128, 8, io=torch.bfloat16, Hk=2, Hv=4, B=2, L=1)
    cw = I.model_weights(w, 9)
    st, cs = I.initial_state(w, 9)
    qkv, g, beta = I.round_stream(w, 0, 9)
    g[0, 0, 2, :, ::5] = 0.0          # channels 0, 5, 10, .. closed at step 2 of sequence 0
    g[0, 1, 0, 1, :64] = 0.0          # head 1 of sequence 1 forgets half its columns at step 0
    g[0, 1, 5, 3, 100:] = 0.0
    r = SpecRound(w)
    dq, dcw, dcs, dg, db, dst = to_dev(qkv, cw, cs, g, beta, st)
    r.verify(dq, dcw, dcs, dg, db, dst)
    r.check_status()
    ref = oracle_verify(w, qkv, cw, cs, g, beta, st)
    assert_close(f64(r.out), ref["out"], "out", bf16=True)
    assert_close(f64(r.tape_delta), ref["tape_delta"], "tape_delta")


@pytest.mark.gpu
def test_gpu_per_channel_gates_full_size_sampled(gdnlib):
    """The --gate-dk workload (30 layers, batch 64, N = 8, g [L, B, T, Hv, 128]) in the bench's
    launch configuration: 8 random (layer, sequence) units of verify compared with the oracle."""
    from parity_util import assert_close, f64, oracle_verify
    from speculative_verify_gdn_gb300 import inputs as I
    from speculative_verify_gdn_gb300.round import SpecRound
    w = I.custom(I.WORKLOADS[2], name=I.WORKLOADS[2].name + "_gdk", gate_dk=True)
    dev = "cuda"
    cw = I.model_weights(w, 0, dev)
    st, cs = I.initial_state(w, 0, dev)
    qkv, g, beta = I.round_stream(w, 0, 0, dev)
    r = SpecRound(w)
    r.verify(qkv, cw, cs, g, beta, st)
    r.check_status()
    rng = np.random.default_rng(17)
    units = {(int(rng.integers(0, w.L)), int(rng.integers(0, w.B))) for _ in range(8)}
    for (l, b) in sorted(units):
        sl = lambda t: t[l:l + 1, b:b + 1].cpu()
        ref = oracle_verify(w, sl(qkv), cw[l:l + 1].cpu(), sl(cs), sl(g), sl(beta), sl(st),
                            L=1, B=1)
        assert_close(f64(r.out[l:l + 1, b:b + 1]), ref["out"], "out (l=%d,b=%d)" % (l, b), bf16=True)
        assert_close(f64(r.tape_delta[l:l + 1, b:b + 1]), ref["tape_delta"], "delta")
        assert_close(f64(r.tape_k[l:l + 1, b:b + 1]), ref["tape_k"], "tape_k")


@pytest.mark.gpu
@pytest.mark.parametrize("D,T", [(128, 8), (64, 4)])
def test_gpu_per_channel_gates_rollback_verify(gdnlib, D, T):
    """gdn_rollback_verify with per-channel gates (served as its two calls) against the oracle's
    rollback followed by its verify."""
    from parity_util import assert_close, f64
    from speculative_verify_gdn_gb300 import inputs as I
    from test_gpu_fused import oracle_commit_then_verify, run_fused
    w = gdk_workload(D, T, io=torch.bfloat16, B=5)
    cw = I.model_weights(w, 3)
    st, cs = I.initial_state(w, 3)
    qkv, g, beta = I.round_stream(w, 1, 3)
    prev = I.previous_round(w, 3)
    assert prev[3].shape == g.shape
    n = np.array([0, T, 1, 2, T // 2], np.int32)
    dst, dcs, out, tdl, tk, status = run_fused(w, n, prev, qkv, cw, cs, g, beta, st)
    assert int(status.item()) == 0
    st1, cs1, bad, ref = oracle_commit_then_verify(w, n, prev, qkv, cw, cs, g, beta, st)
    assert bad == 0
    assert_close(f64(dst), st1, "committed state")
    assert np.array_equal(f64(dcs), cs1)
    assert_close(f64(out), ref["out"], "out", bf16=True)
    assert_close(f64(tdl), ref["tape_delta"], "tape_delta")
    assert_close(f64(tk), ref["tape_k"], "tape_k")


def random_parents(rng, B, T, depth):
    """parent[b][v] in [-1, v): a chain of `depth` nodes first, the rest attached at random to a
    node of depth < depth (or to the context)."""
    par = np.full((B, T), -1, np.int32)
    for b in range(B):
        dep = [0] * T
        for v in range(T):
            if v < depth:
                par[b, v] = v - 1
            else:
                cand = [-1] + [x for x in range(v) if dep[x] < depth - 1]
                par[b, v] = cand[rng.integers(len(cand))]
            dep[v] = 0 if par[b, v] < 0 else dep[par[b, v]] + 1
    return par


@pytest.mark.gpu
@pytest.mark.parametrize("D,T,io", [(32, 8, torch.float32), (64, 16, torch.float32),
                                    (128, 16, torch.float32), (128, 32, torch.bfloat16),
                                    (128, 12, torch.bfloat16)])
def test_gpu_per_channel_gates_trees_and_path_rollback(gdnlib, D, T, io):
    """Trees with one gate per key channel (per-head kernel), then the path rollback along each
    sequence's accepted root-to-leaf prefix, against the oracle's node-by-node recurrence."""
    from parity_util import assert_close, f64, oracle_rollback, oracle_verify, to_dev
    from speculative_verify_gdn_gb300 import inputs as I
    from speculative_verify_gdn_gb300.round import SpecRound
    rng = np.random.default_rng(D + T)
    w = gdk_workload(D, T, io=io, B=3)
    w = I.custom(w, name=w.name + "_tree", accept="tree", tree_depth=min(T, 6), tree_branch=3)
    cw = I.model_weights(w, 5)
    st, cs = I.initial_state(w, 5)
    qkv, g, beta = I.round_stream(w, 0, 5)
    par = torch.from_numpy(random_parents(rng, w.B, T, min(T, 6)))
    r = SpecRound(w)
    dq, dcw, dcs, dg, db, dst = to_dev(qkv, cw, cs, g, beta, st)
    r.verify(dq, dcw, dcs, dg, db, dst, parent=par.cuda())
    r.check_status()
    ref = oracle_verify(w, qkv, cw, cs, g, beta, st, parent=par)
    assert_close(f64(r.out), ref["out"], "out", bf16=io == torch.bfloat16)
    assert_close(f64(r.tape_delta), ref["tape_delta"], "tape_delta")
    assert_close(f64(r.tape_k), ref["tape_k"], "tape_k")
    # accepted paths: the deepest chain from the root (nodes 0, 1, ...) cut at various lengths
    P = r.path.shape[1]
    path = np.zeros((w.B, P), np.int32)
    n = np.array([min(P, 3), 0, P], np.int32)
    for b in range(w.B):
        x, chain = int(np.argmax([len(list(_ancestors(par[b].numpy(), v))) for v in range(T)])), []
        chain = list(_ancestors(par[b].numpy(), x))[::-1][:P]
        path[b, :len(chain)] = chain
        n[b] = min(n[b], len(chain))
    r.path.copy_(torch.from_numpy(path))
    r.n_acc.copy_(torch.from_numpy(n))
    r.rollback(dq, dg, dst, dcs)
    r.check_status()
    st_ref, cs_ref, bad = oracle_rollback(w, n, ref, g, qkv, st, cs, path=path)
    assert bad == 0
    assert_close(f64(dst), st_ref, "state")
    assert np.array_equal(f64(dcs), cs_ref)


def _ancestors(par, v):
    while v >= 0:
        yield v
        v = int(par[v])

