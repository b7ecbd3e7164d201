"""Chain rollback against the oracle where few or no sequences commit (the sampling workloads'
usual round), in large batches, with counts outside [0, T] beside valid ones, and at the full-size
N = 16 sampling shape with a sparse commit pattern."""
import numpy as np
import pytest
import torch

from speculative_verify_gdn_gb300 import inputs as I
from speculative_verify_gdn_gb300.round import SpecRound
from parity_util import assert_close, f64, oracle_rollback, oracle_verify, to_dev
from test_gpu_parity import run_verify_case, small

pytestmark = pytest.mark.gpu


def sparse_counts(B, T, live, seed):
    rng = np.random.default_rng(seed)
    n = np.zeros(B, np.int32)
    for b in live:
        n[b] = int(rng.integers(1, T + 1))
    return n


def rollback_case(w, n, seed=0):
    r, ref, host, dev = run_verify_case(w, seed=seed)
    qkv, cw, cs, g, beta, st = host
    dq, dcw, dcs, dg, db, dst = dev
    r.n_acc.copy_(torch.from_numpy(n))
    r.rollback(dq, dg, dst, dcs)
    return r, ref, host, (dst, dcs)


@pytest.mark.parametrize("B,live", [
    (40, [7]),                           # one sequence commits
    (300, [0, 137, 255, 256, 299]),
    (513, list(range(0, 513, 9))),       # every ninth sequence
])
@pytest.mark.parametrize("D,T", [(32, 4), (128, 8)])
def test_sparse_commits_match_oracle(gdnlib, B, live, D, T):
    L = 2 if D == 32 else 1
    w = small(I.WORKLOADS[1], L=L, B=B, N=T, Hk=1, Hv=2, D=D, W=4, V=64)
    n = sparse_counts(B, T, live, seed=B + D)
    r, ref, (qkv, cw, cs, g, beta, st), (dst, dcs) = rollback_case(w, n, seed=B)
    r.check_status()
    st_ref, cs_ref, bad = oracle_rollback(w, n, ref, g, qkv, st, cs)
    assert bad == 0
    assert_close(f64(dst), st_ref, "state")
    assert np.array_equal(f64(dcs), cs_ref)
    # sequences that accepted nothing keep their snapshot bit for bit
    idle = np.flatnonzero(n == 0)
    assert torch.equal(dst[:, idle].cpu(), st[:, idle])
    assert torch.equal(dcs[:, idle].cpu(), cs[:, idle])


def test_no_commit_is_a_no_op(gdnlib):
    w = small(I.WORKLOADS[1], L=2, B=64, N=8, Hk=2, Hv=4, D=128, W=4, V=64)
    n = np.zeros(64, np.int32)
    r, ref, (qkv, cw, cs, g, beta, st), (dst, dcs) = rollback_case(w, n)
    r.check_status()
    assert torch.equal(dst.cpu(), st) and torch.equal(dcs.cpu(), cs)


@pytest.mark.parametrize("B", [1024, 1025])
def test_large_batches(gdnlib, B):
    w = small(I.WORKLOADS[1], L=1, B=B, N=3, Hk=1, Hv=1, D=32, W=2, V=64)
    n = sparse_counts(B, 3, list(range(0, B, 5)) + [B - 1], seed=B)
    r, ref, (qkv, cw, cs, g, beta, st), (dst, dcs) = rollback_case(w, n, seed=B)
    r.check_status()
    st_ref, cs_ref, bad = oracle_rollback(w, n, ref, g, qkv, st, cs)
    assert bad == 0
    assert_close(f64(dst), st_ref, "state")
    assert np.array_equal(f64(dcs), cs_ref)


def test_bad_counts_beside_valid_ones(gdnlib):
    """Counts outside [0, T] set BAD_NACC and leave their sequences untouched; the valid ones in
    the same call still commit."""
    T = 4
    w = small(I.WORKLOADS[1], L=2, B=6, N=T, Hk=2, Hv=4, D=64, W=4, V=64)
    n = np.array([-1, 2, T + 1, 0, T, 1], np.int32)
    r, ref, (qkv, cw, cs, g, beta, st), (dst, dcs) = rollback_case(w, n)
    torch.cuda.synchronize()
    assert int(r.status.item()) & 0x1
    ok = np.array([1, 3, 4, 5])
    n_ok = np.where(np.isin(np.arange(6), ok), n, 0).astype(np.int32)
    st_ref, cs_ref, bad = oracle_rollback(w, n_ok, ref, g, qkv, st, cs)
    assert_close(f64(dst), st_ref, "state")
    assert np.array_equal(f64(dcs), cs_ref)
    for b in (0, 2):
        assert torch.equal(dst[:, b].cpu(), st[:, b]) and torch.equal(dcs[:, b].cpu(), cs[:, b])


def test_full_size_sampling_shape_sparse_commit(gdnlib):
    """The N = 16 sampling workload's shape (30 layers, batch 16, 32 value heads, d = 128): two
    sequences commit; every layer of both is compared with the oracle, and the others must be
    bit-identical to the snapshot."""
    w = I.WORKLOADS[3]
    dev = "cuda"
    cw = I.model_weights(w, 0, dev)
    st, cs = I.initial_state(w, 0, dev)
    qkv, g, beta = I.round_stream(w, 0, 0, dev)
    st0, cs0 = st.clone(), cs.clone()
    r = SpecRound(w)
    r.verify(qkv, cw, cs, g, beta, st)
    n = np.zeros(w.B, np.int32)
    n[3], n[12] = 1, w.N
    r.n_acc.copy_(torch.from_numpy(n))
    r.rollback(qkv, g, st, cs)
    r.check_status()
    idle = np.flatnonzero(n == 0)
    assert torch.equal(st[:, idle], st0[:, idle]) and torch.equal(cs[:, idle], cs0[:, idle])
    for b in (3, 12):
        for l in range(0, w.L, 7):
            sl = lambda t: t[l:l + 1, b:b + 1].cpu()
            ref = oracle_verify(w, sl(qkv), cw[l:l + 1].cpu(), sl(cs0), sl(g), sl(beta), sl(st0),
                                L=1, B=1)
            st_ref, cs_ref, bad = oracle_rollback(w, n[b:b + 1], ref, sl(g), sl(qkv), sl(st0),
                                                  sl(cs0), L=1, B=1)
            assert bad == 0
            assert_close(f64(st[l:l + 1, b:b + 1]), st_ref, "state (l=%d,b=%d)" % (l, b))
            assert np.array_equal(f64(cs[l:l + 1, b:b + 1]), cs_ref)
