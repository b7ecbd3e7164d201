"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs.

Small shapes are compared in full; the full-size workloads are compared on sampled
(layer, sequence) units plus every accept output, with inputs drawn on the device (seeded) and the
sampled slices copied to the host for the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_verify_gdn_gb300 import _lib, inputs as I
from speculative_verify_gdn_gb300.round import SpecRound
from parity_util import (assert_close, f64, logits_f32, oracle_rollback, oracle_verify, to_dev)

pytestmark = pytest.mark.gpu


def small(base, **kw):
    kw.setdefault("name", "small_" + "_".join("%s%s" % (k, v) for k, v in sorted(kw.items())))
    return I.custom(base, **kw)


def is_bf16(t):
    return t.dtype == torch.bfloat16


def make_model(w, seed=0, device="cpu"):
    cw = I.model_weights(w, seed, device)
    st, cs = I.initial_state(w, seed, device)
    return cw, st, cs


def run_verify_case(w, seed=0, parent=None):
    cw, st, cs = make_model(w, seed)
    qkv, g, beta = I.round_stream(w, 0, seed)
    r = SpecRound(w)
    dq, dcw, dcs, dg, db, dst = to_dev(qkv, cw, cs, g, beta, st)
    dpar = None if parent is None else parent.cuda()
    r.verify(dq, dcw, dcs, dg, db, dst, parent=dpar)
    r.check_status()
    ref = oracle_verify(w, qkv, cw, cs, g, beta, st, parent=parent)
    assert_close(f64(r.out), ref["out"], "out", bf16=is_bf16(r.out))
    assert_close(f64(r.tape_delta), ref["tape_delta"], "tape_delta")
    assert_close(f64(r.tape_k), ref["tape_k"], "tape_k")
    # the snapshot is untouched
    assert torch.equal(dst.cpu(), st) and torch.equal(dcs.cpu(), cs)
    return r, ref, (qkv, cw, cs, g, beta, st), (dq, dcw, dcs, dg, db, dst)


# ------------------------------------------------------------------------------ verify
def test_verify_tiny_workload(gdnlib):
    run_verify_case(I.WORKLOADS[0])


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("T", [1, 3, 4, 5, 8, 13, 16, 32])
def test_verify_shapes(gdnlib, D, T):
    w = small(I.WORKLOADS[1], L=2, B=3, N=T, Hk=2, Hv=4, D=D, W=4, V=64)
    run_verify_case(w, seed=T * 7 + D)


@pytest.mark.parametrize("W", [1, 2, 3])
@pytest.mark.parametrize("io", [torch.float32, torch.bfloat16])
def test_verify_conv_widths_and_dtypes(gdnlib, W, io):
    w = small(I.WORKLOADS[1], L=1, B=2, N=6, Hk=1, Hv=3, D=32, W=W, V=64, io_dtype=io)
    run_verify_case(w, seed=W)


@pytest.mark.parametrize("Hk,Hv,T", [(4, 4, 8), (3, 6, 2), (1, 2, 7), (2, 2, 16), (2, 4, 12), (1, 1, 9)])
def test_verify_head_groupings(gdnlib, Hk, Hv, T):
    """One and two value heads per key head at d = 128 (both layouts of the pipelined kernel)."""
    w = small(I.WORKLOADS[1], L=2, B=3, N=T, Hk=Hk, Hv=Hv, D=128, V=64)
    run_verify_case(w, seed=Hk * 10 + Hv)


def test_verify_qwen36_b1(gdnlib):
    """The 30-layer Qwen3.6-shaped stack at batch 1, N = 4, every output compared."""
    run_verify_case(I.WORKLOADS[1])


def test_verify_empty_is_noop(gdnlib):
    sh = _lib.GdnShape(L=1, B=1, T=0, Hk=2, Hv=4, Dk=32, Dv=32, W=4, io_dtype=torch.float32)
    z = lambda *s: torch.zeros(s, device="cuda")
    _lib.verify(sh, z(1, 1, 0, sh.C), z(1, sh.C, 4), z(1, 1, 3, sh.C), z(1, 1, 0, 4),
                z(1, 1, 0, 4), z(1, 1, 4, 32, 32), z(1, 1, 0, 4, 32), z(1, 1, 0, 4, 32),
                z(1, 1, 0, 2, 32))


# ------------------------------------------------------------------------------ rollback
@pytest.mark.parametrize("D,T", [(32, 4), (64, 8), (128, 5), (128, 16), (32, 32)])
def test_rollback_matches_oracle(gdnlib, D, T):
    w = small(I.WORKLOADS[1], L=2, B=5, N=T, Hk=2, Hv=4, D=D, W=4, V=64)
    r, ref, host, dev = run_verify_case(w, seed=D + T)
    qkv, cw, cs, g, beta, st = host
    dq, dcw, dcs, dg, db, dst = dev
    n = np.array([0, T, 1, min(2, T), T // 2], np.int32)
    r.n_acc.copy_(torch.from_numpy(n))
    r.rollback(dq, dg, dst, dcs)
    r.check_status()
    st_ref, cs_ref, bad = oracle_rollback(w, n, ref, g, qkv, st, cs)
    assert bad == 0
    assert_close(f64(dst), st_ref, "state")
    # the conv state is a copy of raw rows: exact
    assert np.array_equal(f64(dcs), cs_ref)
    # n = 0 leaves the snapshot bit-identical
    assert torch.equal(dst[:, 0].cpu(), st[:, 0])


@pytest.mark.parametrize("D,T,W", [(128, 8, 1), (128, 8, 2), (64, 6, 3), (32, 16, 2)])
def test_rollback_conv_widths(gdnlib, D, T, W):
    """Shorter conv windows: fewer conv-state rows rebuilt (W - 1 of them, none for W = 1)."""
    w = small(I.WORKLOADS[1], L=2, B=4, N=T, Hk=2, Hv=4, D=D, W=W, V=64)
    r, ref, host, dev = run_verify_case(w, seed=3 * W + T)
    qkv, cw, cs, g, beta, st = host
    dq, dcw, dcs, dg, db, dst = dev
    n = np.array([T, 1, 0, T - 1], np.int32)
    r.n_acc.copy_(torch.from_numpy(n))
    r.rollback(dq, dg, dst, dcs)
    r.check_status()
    st_ref, cs_ref, bad = oracle_rollback(w, n, ref, g, qkv, st, cs)
    assert bad == 0
    assert_close(f64(dst), st_ref, "state")
    assert np.array_equal(f64(dcs), cs_ref)


def test_rollback_path_bad_node_sets_status_and_skips(gdnlib):
    """A path entry outside [0, T) is reported and that sequence's state is left as it was; the
    other sequence commits normally."""
    w, par = tree_case(B=2, T=8, D=128, depth=4)
    r, ref, host, dev = run_verify_case(w, parent=par)
    qkv, cw, cs, g, beta, st = host
    dq, dcw, dcs, dg, db, dst = dev
    path = np.zeros((w.B, r.path.shape[1]), np.int32)
    path[0, :2] = [0, 1]
    path[1, :2] = [0, 9]                       # node 9 does not exist (T = 8)
    r.path.copy_(torch.from_numpy(path))
    r.n_acc.copy_(torch.tensor([2, 2], dtype=torch.int32))
    before = dst.clone()
    r.rollback(dq, dg, dst, dcs)
    torch.cuda.synchronize()
    assert int(r.status.item()) & 0x8
    assert torch.equal(dst[:, 1].cpu(), before[:, 1].cpu())
    st_ref, _, bad = oracle_rollback(w, np.array([2, 0], np.int32), ref, g, qkv, st, cs,
                                     path=path)
    assert_close(f64(dst[:, :1]), st_ref[:, :1], "state of the valid sequence")


def test_rollback_bad_count_sets_status_and_skips(gdnlib):
    w = small(I.WORKLOADS[1], L=1, B=2, N=4, Hk=2, Hv=4, D=32, V=64)
    r, ref, host, dev = run_verify_case(w)
    dq, dcw, dcs, dg, db, dst = dev
    before = dst.clone()
    r.n_acc.copy_(torch.tensor([5, -1], dtype=torch.int32))
    r.rollback(dq, dg, dst, dcs)
    torch.cuda.synchronize()
    assert int(r.status.item()) & 0x1
    assert torch.equal(before, dst)


# ------------------------------------------------------------------------------ greedy accept
@pytest.mark.parametrize("wid", [0, 1])
def test_greedy_accept_bit_exact(gdnlib, wid):
    w = I.WORKLOADS[wid]
    r = SpecRound(w)
    for rnd in range(8):
        lg, dr, L = I.greedy_logits(w, rnd)
        dlg, ddr = to_dev(lg, dr)
        r.accept(dlg, ddr, round_=rnd)
        r.check_status()
        n, out, bad = oracle.accept_greedy(logits_f32(lg), dr.numpy())
        assert np.array_equal(r.n_acc.cpu().numpy(), n)
        assert np.array_equal(r.out_tokens.cpu().numpy(), out)
        assert np.array_equal(n, L.numpy())


@pytest.mark.parametrize("V", [1000, 1003, 8191, 151936])
def test_greedy_accept_ties_and_ragged_vocab(gdnlib, V):
    torch.manual_seed(V)
    B, N = 7, 5
    Vpad = (V + 7) // 8 * 8
    lg = torch.randint(-3, 3, (B, N + 1, Vpad)).to(torch.bfloat16)   # many exact ties
    lg[..., V:] = 100                                                   # padding never read
    am = lg[..., :V].float().argmax(-1)
    dr = am[:, :N].clone().to(torch.int32)
    dr[1, 0] = (dr[1, 0] + 1) % V
    dr[3, 2] = (dr[3, 2] + 1) % V
    ws = torch.empty(_lib.workspace_bytes(B, N, V), dtype=torch.uint8, device="cuda")
    n_acc = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, N + 1, dtype=torch.int32, device="cuda")
    dlg, ddr = to_dev(lg, dr)
    _lib.spec_accept(dlg, ddr, n_acc, out, ws, V=V)
    torch.cuda.synchronize()
    n_ref, out_ref, _ = oracle.accept_greedy(logits_f32(lg[..., :V].contiguous()), dr.numpy())
    assert np.array_equal(n_acc.cpu().numpy(), n_ref)
    assert np.array_equal(out.cpu().numpy(), out_ref)


def test_accept_bad_draft_token(gdnlib):
    w = small(I.WORKLOADS[0], B=3, name="bad_tok")
    r = SpecRound(w)
    lg, dr, _ = I.greedy_logits(w, 0)
    dr[1, 2] = w.V + 5
    dlg, ddr = to_dev(lg, dr)
    r.accept(dlg, ddr)
    torch.cuda.synchronize()
    assert int(r.status.item()) & 0x4
    n_ref, out_ref, bad = oracle.accept_greedy(logits_f32(lg), dr.numpy())
    assert bad == 4
    assert np.array_equal(r.n_acc.cpu().numpy(), n_ref)
    assert np.array_equal(r.out_tokens.cpu().numpy(), out_ref)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_accept_nan_logits(gdnlib, dtype):
    """NaN logits count as −∞ on both sides: greedy never picks one (a row of NaN / −∞ gives
    index 0), sampling gives it weight 0. Token ids and counts bit-exact with the oracle."""
    B, N, V = 8, 3, 1000
    gen = torch.Generator().manual_seed(5)
    lg = torch.randn(B, N + 1, V, generator=gen).to(dtype)
    nan, inf = float("nan"), float("inf")
    lg[0, 0, 0] = nan
    lg[0, 1, :17] = nan
    lg[1, 0, int(lg[1, 0].float().argmax())] = nan       # the maximum itself becomes NaN
    lg[2, 2, :] = nan                                     # a whole NaN row
    lg[3, 1, :] = -inf
    lg[3, 1, 500:] = nan                                  # a row of −∞ and NaN
    lg[4, 3, 1::2] = nan
    lg[5, :, 900:] = nan                                  # NaN tail across the chunks
    lf = logits_f32(lg)
    am = np.array([[oracle.argmax(lf[b, i]) for i in range(N + 1)] for b in range(B)])
    dr = torch.from_numpy(am[:, :N].astype(np.int32))
    dr[6, 1] = (dr[6, 1] + 1) % V
    dlg, ddr = to_dev(lg, dr)
    n_acc = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, N + 1, dtype=torch.int32, device="cuda")
    ws = torch.empty(_lib.workspace_bytes(B, N, V, _lib.SPEC_MODE_GREEDY, dtype), dtype=torch.uint8,
                     device="cuda")
    _lib.spec_accept(dlg, ddr, n_acc, out, ws)
    torch.cuda.synchronize()
    n_ref, out_ref, _ = oracle.accept_greedy(lf, dr.numpy())
    assert np.array_equal(n_acc.cpu().numpy(), n_ref)
    assert np.array_equal(out.cpu().numpy(), out_ref)
    ws = torch.empty(_lib.workspace_bytes(B, N, V, _lib.SPEC_MODE_SAMPLE, dtype), dtype=torch.uint8,
                     device="cuda")
    for rnd in range(4):
        _lib.spec_accept(dlg, ddr, n_acc, out, ws, mode=_lib.SPEC_MODE_SAMPLE, temperature=0.7,
                         seed=13, round_=rnd)
        torch.cuda.synchronize()
        n_ref, out_ref, _ = oracle.accept_sample(lf, dr.numpy(), 0.7, 13, rnd)
        assert np.array_equal(n_acc.cpu().numpy(), n_ref)
        assert np.array_equal(out.cpu().numpy(), out_ref)
        tok = out.cpu().numpy()
        for b in range(B):
            for i in range(N + 1):
                if tok[b, i] >= 0:
                    assert not np.isnan(lf[b, i, tok[b, i]])


# ------------------------------------------------------------------------------ sampling accept
@pytest.mark.parametrize("V,B,N", [(4096, 16, 16), (151936, 16, 16), (1000, 5, 0), (333, 9, 3)])
def test_sample_accept_bit_exact(gdnlib, V, B, N):
    w = I.custom(I.WORKLOADS[3], name="samp_%d_%d_%d" % (V, B, N), V=V, B=B, N=N, L=1)
    Vpad = (V + 7) // 8 * 8
    ws = torch.empty(_lib.workspace_bytes(B, N, V, _lib.SPEC_MODE_SAMPLE), dtype=torch.uint8,
                     device="cuda")
    n_acc = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, N + 1, dtype=torch.int32, device="cuda")
    for rnd in range(3):
        lg, dr = I.sample_logits(w, rnd)
        # perturb some drafts away from the argmax so both accept and reject paths run
        dr[::2, ::3] = (dr[::2, ::3] + 1) % V
        pad = torch.full((B, N + 1, Vpad), 50.0).to(lg.dtype)     # padding is never read
        pad[..., :V] = lg
        dlg, ddr = to_dev(pad, dr)
        _lib.spec_accept(dlg, ddr, n_acc, out, ws, mode=_lib.SPEC_MODE_SAMPLE,
                         temperature=w.temperature, seed=77, round_=rnd, V=V)
        torch.cuda.synchronize()
        n, out_ref, bad = oracle.accept_sample(logits_f32(lg), dr.numpy(), w.temperature, 77, rnd)
        assert bad == 0
        assert np.array_equal(n_acc.cpu().numpy(), n)
        assert np.array_equal(out.cpu().numpy(), out_ref)


def sample_case(B, N, V, dtype, temperature, seed, rounds, plant=None, std=2.0):
    """Sampling accept through the C ABI against the oracle, bit-exact, over `rounds` rounds.
    Rows are padded to a 16-byte stride with values that must never be read. `plant(lg, dr, g)`
    may edit the logits / drafts (a numpy generator is passed)."""
    g = np.random.default_rng(seed)
    VN = 8 if dtype == torch.bfloat16 else 4
    Vpad = (V + VN - 1) // VN * VN
    ws = torch.empty(_lib.workspace_bytes(B, N, V, _lib.SPEC_MODE_SAMPLE, dtype), dtype=torch.uint8,
                     device="cuda")
    n_acc = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, N + 1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lengths = []
    for rnd in range(rounds):
        lg = torch.from_numpy((g.standard_normal((B, N + 1, V)) * std).astype(np.float32))
        dr = lg[:, :N].argmax(-1).to(torch.int32)
        if plant is not None:
            plant(lg, dr, g)
        lg = lg.to(dtype)
        pad = torch.full((B, N + 1, Vpad), 1e4).to(dtype)       # padding is never read
        pad[..., :V] = lg
        dlg, ddr = to_dev(pad, dr)
        _lib.spec_accept(dlg, ddr, n_acc, out, ws, mode=_lib.SPEC_MODE_SAMPLE,
                         temperature=temperature, seed=seed, round_=rnd, V=V, status=status)
        torch.cuda.synchronize()
        n, out_ref, bad = oracle.accept_sample(logits_f32(lg), dr.numpy(), temperature, seed, rnd)
        assert bad == 0
        assert np.array_equal(n_acc.cpu().numpy(), n), (rnd, n_acc.cpu().numpy(), n)
        assert np.array_equal(out.cpu().numpy(), out_ref), rnd
        lengths += list(n)
    assert int(status.item()) == 0
    return np.array(lengths)


# vocabularies on both sides of the switch between the parallel three-kernel path (V < 8192, or
# two rows' slices beyond shared memory: fp32 above ~230K) and the one-cluster-per-sequence path;
# ragged slices and runs; batch sizes that need one and several waves of clusters
@pytest.mark.parametrize("V,dtype,B", [(8192, torch.bfloat16, 5), (8191, torch.bfloat16, 5),
                                       (50001, torch.bfloat16, 5), (262147, torch.bfloat16, 3),
                                       (151936, torch.float32, 5), (163841, torch.float32, 4),
                                       (262144, torch.float32, 2), (12345, torch.float32, 7),
                                       (151936, torch.bfloat16, 37), (20000, torch.bfloat16, 200)])
def test_sample_accept_vocab_sizes(gdnlib, V, dtype, B):
    sample_case(B=B, N=3, V=V, dtype=dtype, temperature=0.7, seed=V % 97, rounds=2)


def test_sample_accept_long_accept_runs(gdnlib):
    """Drafts that carry most of the probability (a planted margin at low temperature) are
    accepted for many rows in a row, so the cluster walks deep into the block and often reaches
    the bonus row; a few rows plant a rejection at a random depth."""
    B, N, V = 12, 16, 151936

    def plant(lg, dr, g):
        for b in range(B):
            stop = int(g.integers(0, N + 3))            # >= N: no planted rejection
            for i in range(N):
                d = int(g.integers(0, V))
                dr[b, i] = d
                lg[b, i, d] = lg[b, i].max() + (4.0 if i != stop else -3.0)

    n = sample_case(B=B, N=N, V=V, dtype=torch.bfloat16, temperature=0.5, seed=21, rounds=3,
                    plant=plant)
    assert n.max() == N and (n > N // 2).mean() > 0.3


def test_sample_accept_zero_draft_rows(gdnlib):
    """N = 0: only the bonus row, sampled by the cluster path."""
    sample_case(B=9, N=0, V=151936, dtype=torch.bfloat16, temperature=1.3, seed=5, rounds=3)


def test_sample_accept_bad_draft_on_cluster_path(gdnlib):
    """A draft outside [0, V) on the cluster path: that sequence reports n = 0 and -1 tokens with
    BAD_TOKEN (its CTAs leave once their row copies have landed); the others are unaffected."""
    B, N, V = 6, 5, 151936
    g = np.random.default_rng(8)
    lg = torch.from_numpy((g.standard_normal((B, N + 1, V)) * 2).astype(np.float32)).to(torch.bfloat16)
    dr = lg[:, :N].float().argmax(-1).to(torch.int32)
    dr[2, 3] = V + 1
    dr[4, 0] = -7
    ws = torch.empty(_lib.workspace_bytes(B, N, V, _lib.SPEC_MODE_SAMPLE), dtype=torch.uint8,
                     device="cuda")
    n_acc = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, N + 1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dlg, ddr = to_dev(lg, dr)
    _lib.spec_accept(dlg, ddr, n_acc, out, ws, mode=_lib.SPEC_MODE_SAMPLE, temperature=0.7,
                     seed=3, round_=1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x4
    n, out_ref, bad = oracle.accept_sample(logits_f32(lg), dr.numpy(), 0.7, 3, 1)
    assert bad == 4
    assert np.array_equal(n_acc.cpu().numpy(), n)
    assert np.array_equal(out.cpu().numpy(), out_ref)
    assert (out_ref[2] == -1).all() and (out_ref[4] == -1).all()


def test_sample_accept_chi_square_gpu(gdnlib):
    """Emitted first tokens follow p over 10^6 GPU draws (all sequences share one logits block)."""
    from scipy import stats
    V, T, Bn = 48, 0.7, 1_000_000
    g = np.random.default_rng(3)
    lg = torch.from_numpy((g.standard_normal((1, 2, V)) * 2).astype(np.float32))
    p = np.exp((lg[0, 0].double().numpy() - lg[0, 0].double().numpy().max()) / np.float32(T))
    p /= p.sum()
    dr = torch.from_numpy(g.integers(0, V, (Bn, 1)).astype(np.int32))
    ws = torch.empty(_lib.workspace_bytes(Bn, 1, V, _lib.SPEC_MODE_SAMPLE, torch.float32),
                     dtype=torch.uint8, device="cuda")
    n_acc = torch.empty(Bn, dtype=torch.int32, device="cuda")
    out = torch.empty(Bn, 2, dtype=torch.int32, device="cuda")
    _lib.spec_accept(lg.cuda(), dr.cuda(), n_acc, out, ws, mode=_lib.SPEC_MODE_SAMPLE,
                     temperature=T, seed=99, round_=4, broadcast_B=Bn)
    first = out[:, 0].cpu().numpy()
    counts = np.bincount(first, minlength=V)
    exp = p * Bn
    keep = exp >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    ex = np.append(exp[keep], exp[~keep].sum())
    assert stats.chisquare(obs, ex * obs.sum() / ex.sum()).pvalue > 1e-3
    # the same draws as the oracle on a subset
    n_o, out_o, _ = oracle.accept_sample(lg.numpy(), dr.numpy()[:5000], T, 99, 4,
                                         seq_shared=True, B=5000)
    assert np.array_equal(out.cpu().numpy()[:5000], out_o)


# ------------------------------------------------------------------------------ tree
def tree_case(B=3, T=12, D=32, L=2, depth=5, seed=0, Hv=4, branch=None):
    kw = {} if branch is None else {"tree_branch": branch}
    w = I.custom(I.WORKLOADS[4], name="tree_%d_%d_%d_%d_%d" % (B, T, D, Hv, depth), L=L, B=B,
                 N=T, Hk=2, Hv=Hv, D=D, V=512, tree_depth=depth, **kw)
    par = I.random_tree(w, 0, seed)
    return w, par


# D = 128 bf16 trees run on the pipelined kernel (node counts up to 8, 16 and 32, one and two
# value heads per key head, ragged counts; 17 nodes is the smallest tree of the 32-node kernel, and
# depth 16 takes its solve's path longer than its 8 register slots); the others on the per-head kernel
@pytest.mark.parametrize("T,D,Hv,depth", [(12, 32, 4, 8), (32, 64, 4, 8), (7, 128, 4, 7),
                                          (16, 128, 4, 8), (13, 128, 2, 5), (32, 128, 4, 8),
                                          (32, 128, 2, 6), (24, 128, 4, 3), (29, 128, 2, 12),
                                          (17, 128, 4, 6), (32, 128, 4, 16)])
def test_tree_verify_matches_oracle(gdnlib, T, D, Hv, depth):
    w, par = tree_case(T=T, D=D, depth=depth, Hv=Hv, B=4)
    run_verify_case(w, parent=par)


@pytest.mark.parametrize("T,tree,Hv", [(16, False, 4), (16, False, 8), (32, True, 4), (32, True, 8)])
def test_pipe_several_units_per_cta(gdnlib, T, tree, Hv):
    """More units than SMs (320 (layer, sequence, key head) units), so each CTA of the pipelined
    kernel runs two or three in turn: every per-unit barrier phase, including the epilogue's
    tensor-core solve of 16-position chains and 32-node trees, with one and two value heads per
    key head."""
    if tree:
        w = I.custom(I.WORKLOADS[4], name="tree_many_%d_%d" % (T, Hv), L=1, B=80, N=T, Hk=4,
                     Hv=Hv, D=128, V=64, tree_depth=8)
        run_verify_case(w, parent=I.random_tree(w, 0, 0))
    else:
        run_verify_case(small(I.WORKLOADS[1], L=1, B=80, N=T, Hk=4, Hv=Hv, D=128, V=64), seed=5)


@pytest.mark.parametrize("shape", ["chain", "star"])
def test_tree_verify_degenerate_trees(gdnlib, shape):
    """A tree that is one chain (every node the child of the one before) equals the chain
    verify; a star (every node a child of the context) starts every node from S_0."""
    T = 32
    w, _ = tree_case(T=T, D=128, depth=T if shape == "chain" else 1, B=3, branch=T)
    par = torch.arange(-1, T - 1, dtype=torch.int32) if shape == "chain" else \
        torch.full((T,), -1, dtype=torch.int32)
    run_verify_case(w, parent=par.repeat(w.B, 1).contiguous())


def test_tree_accept_and_path_rollback(gdnlib):
    w, par = tree_case(B=4, T=20, D=32, depth=6)
    r, ref, host, dev = run_verify_case(w, parent=par)
    qkv, cw, cs, g, beta, st = host
    dq, dcw, dcs, dg, db, dst = dev
    tok, lg, Ls = I.tree_tokens_and_logits(w, par, 0)
    dpar, dtok, dlg = to_dev(par, tok, lg)
    r.accept(dlg, dtok, parent=dpar)
    r.check_status()
    path, n, out, bad = oracle.accept_tree(logits_f32(lg), par.numpy(), tok.numpy(), w.P)
    assert bad == 0
    assert np.array_equal(n, Ls.numpy())
    assert np.array_equal(r.n_acc.cpu().numpy(), n)
    assert np.array_equal(r.path.cpu().numpy(), path)
    assert np.array_equal(r.out_tokens.cpu().numpy(), out)
    r.rollback(dq, dg, dst, dcs)
    r.check_status()
    st_ref, cs_ref, bad = oracle_rollback(w, n, ref, g, qkv, st, cs, path=path)
    assert bad == 0
    assert_close(f64(dst), st_ref, "state")
    assert np.array_equal(f64(dcs), cs_ref)


@pytest.mark.parametrize("T,D", [(6, 32), (20, 128)])
def test_tree_bad_parent_sets_status(gdnlib, T, D):
    w, par = tree_case(B=2, T=T, D=D, depth=4)
    par = par.clone()
    par[1, 3] = 5            # parent after the node
    cw, st, cs = make_model(w)
    qkv, g, beta = I.round_stream(w, 0)
    r = SpecRound(w)
    dq, dcw, dcs, dg, db, dst = to_dev(qkv, cw, cs, g, beta, st)
    r.verify(dq, dcw, dcs, dg, db, dst, parent=par.cuda())
    torch.cuda.synchronize()
    assert int(r.status.item()) & 0x2


# ------------------------------------------------------------------------------ multi-round
def test_three_rounds_small_stack(gdnlib):
    """verify -> accept -> rollback chained over rounds, state carried on both sides."""
    w = small(I.WORKLOADS[2], L=3, B=6, N=8, Hk=2, Hv=4, D=64, V=2048, name="rounds3")
    cw, st, cs = make_model(w)
    dcw, dst, dcs = to_dev(cw, st, cs)
    r = SpecRound(w)
    st_ref, cs_ref = f64(st), f64(cs)
    for rnd in range(3):
        qkv, g, beta = I.round_stream(w, rnd)
        lg, dr, L = I.greedy_logits(w, rnd)
        dq, dg, db, dlg, ddr = to_dev(qkv, g, beta, lg, dr)
        r.step(dq, dg, db, dlg, ddr, dcw, dst, dcs, round_=rnd)
        r.check_status()
        d = oracle.OracleDims(L=w.L, B=w.B, T=w.N, Hk=w.Hk, Hv=w.Hv, Dk=w.D, Dv=w.D, W=w.W)
        ref = oracle.verify(d, f64(qkv), f64(cw), cs_ref, f64(g), f64(beta), st_ref)
        n, out, _ = oracle.accept_greedy(logits_f32(lg), dr.numpy())
        assert np.array_equal(r.n_acc.cpu().numpy(), n)
        assert_close(f64(r.out), ref["out"], "out round %d" % rnd, bf16=True)
        st_ref, cs_ref, _ = oracle.rollback(d, n, ref["tape_delta"], ref["tape_k"], f64(g),
                                            f64(qkv), st_ref, cs_ref)
        assert_close(f64(dst), st_ref, "state round %d" % rnd)
        assert_close(f64(dcs), cs_ref, "conv_state round %d" % rnd, rtol=0, atol_frac=0)


# ------------------------------------------------------------------------------ full-size, sampled
@pytest.mark.parametrize("wid", [2, 3, 4])
def test_full_size_round_sampled_units(gdnlib, wid):
    """One round of the full workload in the bench's launch configuration; every accept output is
    compared, and 16 random (layer, sequence) units of verify and rollback."""
    w = I.WORKLOADS[wid]
    dev = "cuda"
    cw = I.model_weights(w, 0, dev)
    st, cs = I.initial_state(w, 0, dev)
    qkv, g, beta = I.round_stream(w, 0, 0, dev)
    parent = tok = None
    if w.accept == "tree":
        parent = I.random_tree(w, 0)
        tok, lg, _ = I.tree_tokens_and_logits(w, parent, 0)
        parent, tok, lg = to_dev(parent, tok, lg)
        drafts = tok
    elif w.accept == "sample":
        lg, drafts = I.sample_logits(w, 0, 0, dev)
    else:
        lg, drafts, _ = I.greedy_logits(w, 0, 0, dev)
    st0, cs0 = st.clone(), cs.clone()
    r = SpecRound(w)
    r.step(qkv, g, beta, lg, drafts, cw, st, cs, round_=0, seed=5, parent=parent)
    r.check_status()
    lgh = logits_f32(lg)
    if w.accept == "tree":
        path, n, out, _ = oracle.accept_tree(lgh, parent.cpu().numpy(), tok.cpu().numpy(), w.P)
        assert np.array_equal(r.path.cpu().numpy(), path)
    elif w.accept == "sample":
        n, out, _ = oracle.accept_sample(lgh, drafts.cpu().numpy(), w.temperature, 5, 0)
        path = None
    else:
        n, out, _ = oracle.accept_greedy(lgh, drafts.cpu().numpy())
        path = None
    assert np.array_equal(r.n_acc.cpu().numpy(), n)
    assert np.array_equal(r.out_tokens.cpu().numpy(), out)
    rng = np.random.default_rng(wid)
    units = {(int(rng.integers(0, w.L)), int(rng.integers(0, w.B))) for _ in range(16)}
    for (l, b) in sorted(units):
        sl = lambda t: t[l:l + 1, b:b + 1].cpu()
        par_b = None if parent is None else parent[b:b + 1].cpu()
        ref = oracle_verify(w, sl(qkv), cw[l:l + 1].cpu(), sl(cs0), sl(g), sl(beta), sl(st0),
                            parent=par_b, L=1, B=1)
        assert_close(f64(r.out[l:l + 1, b:b + 1]), ref["out"], "out (l=%d,b=%d)" % (l, b),
                     bf16=True)
        assert_close(f64(r.tape_delta[l:l + 1, b:b + 1]), ref["tape_delta"], "delta")
        st_ref, cs_ref, bad = oracle_rollback(w, n[b:b + 1], ref, sl(g), sl(qkv), sl(st0),
                                              sl(cs0), path=None if path is None
                                              else path[b:b + 1], L=1, B=1)
        assert bad == 0
        assert_close(f64(st[l:l + 1, b:b + 1]), st_ref, "state (l=%d,b=%d)" % (l, b))
        assert np.array_equal(f64(cs[l:l + 1, b:b + 1]), cs_ref)
