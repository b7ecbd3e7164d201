"""GPU parity of gdn_rollback_verify (the previous round's rollback and this round's verify in one
call) against the oracle's rollback followed by its verify, on seeded synthetic inputs: the
previous round's tape comes from the input generator, never from the CUDA path."""
import numpy as np
import pytest
import torch

import oracle
from speculative_verify_gdn_gb300 import _lib, inputs as I
from speculative_verify_gdn_gb300.round import SpecRound
from parity_util import assert_close, f64, logits_f32, oracle_dims, to_dev

pytestmark = pytest.mark.gpu


def small(base, **kw):
    kw.setdefault("name", "fused_" + "_".join("%s%s" % (k, v) for k, v in sorted(kw.items())
                                              if k != "io_dtype"))
    return I.custom(base, **kw)


def oracle_commit_then_verify(w, n, prev, qkv, cw, cs, g, beta, st, L=None, B=None):
    d = oracle_dims(w, L=L, B=B)
    _, dl, k, gp, qp = prev
    st1, cs1, bad = oracle.rollback(d, np.asarray(n, np.int32), f64(dl), f64(k), f64(gp), f64(qp),
                                    f64(st), f64(cs))
    ref = oracle.verify(d, f64(qkv), f64(cw), cs1, f64(g), f64(beta), st1)
    return st1, cs1, bad, ref


def run_fused(w, n, prev, qkv, cw, cs, g, beta, st, status=None):
    sh = _lib.GdnShape(L=w.L, B=w.B, T=w.N, Hk=w.Hk, Hv=w.Hv, Dk=w.D, Dv=w.D, W=w.W,
                       io_dtype=w.io_dtype, gate_dk=w.gate_dk)
    _, dl, k, gp, qp = prev
    dn, ddl, dk, dgp, dqp, dq, dcw, dcs, dg, db, dst = to_dev(
        torch.as_tensor(n, dtype=torch.int32), dl, k, gp, qp, qkv, cw, cs, g, beta, st)
    out = torch.empty(sh.out_shape(), dtype=w.io_dtype, device="cuda")
    tdl = torch.empty(sh.out_shape(), dtype=torch.float32, device="cuda")
    tk = torch.empty(sh.tape_k_shape(), dtype=torch.float32, device="cuda")
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.rollback_verify(sh, dn, ddl, dk, dgp, dqp, dq, dcw, dcs, dg, db, dst, out, tdl, tk,
                         status=status)
    torch.cuda.synchronize()
    return dst, dcs, out, tdl, tk, status


# (D, T, Hk, Hv, W, io): the pipelined kernel's shapes (bf16, D = 128, T <= 8, Hv in {Hk, 2Hk})
# and shapes served by the two-call path
CASES = [(128, 8, 2, 4, 4, torch.bfloat16), (128, 4, 2, 2, 4, torch.bfloat16),
         (128, 8, 2, 4, 2, torch.bfloat16), (128, 6, 2, 4, 3, torch.bfloat16),
         (128, 3, 2, 2, 1, torch.bfloat16), (128, 8, 1, 2, 4, torch.bfloat16),
         (32, 5, 2, 4, 4, torch.float32), (64, 8, 2, 4, 4, torch.bfloat16),
         (128, 16, 2, 4, 4, torch.bfloat16)]


@pytest.mark.parametrize("D,T,Hk,Hv,W,io", CASES)
def test_rollback_verify_matches_oracle(gdnlib, D, T, Hk, Hv, W, io):
    w = small(I.WORKLOADS[1], L=2, B=6, N=T, Hk=Hk, Hv=Hv, D=D, W=W, V=64, io_dtype=io)
    cw = I.model_weights(w, 3)
    st, cs = I.initial_state(w, 3)
    qkv, g, beta = I.round_stream(w, 1, 3)
    prev = I.previous_round(w, 3)
    # every regime: nothing, everything, fewer and more rows than the conv window, half
    n = np.minimum(np.array([0, T, 1, 2, T // 2, 3], np.int32), T)
    dst, dcs, out, tdl, tk, status = run_fused(w, n, prev, qkv, cw, cs, g, beta, st)
    assert int(status.item()) == 0
    st1, cs1, bad, ref = oracle_commit_then_verify(w, n, prev, qkv, cw, cs, g, beta, st)
    assert bad == 0
    assert_close(f64(dst), st1, "committed state")
    assert np.array_equal(f64(dcs), cs1), "conv state is a copy of raw rows"
    assert_close(f64(out), ref["out"], "out", bf16=io == torch.bfloat16)
    assert_close(f64(tdl), ref["tape_delta"], "tape_delta")
    assert_close(f64(tk), ref["tape_k"], "tape_k")
    # n = 0 leaves that sequence's state bit-identical
    assert torch.equal(dst[:, 0].cpu(), st[:, 0])


def test_rollback_verify_bad_count_commits_nothing(gdnlib):
    w = small(I.WORKLOADS[1], L=2, B=4, N=8, Hk=2, Hv=4, D=128, W=4, V=64,
              io_dtype=torch.bfloat16, name="fused_badcount")
    cw = I.model_weights(w, 4)
    st, cs = I.initial_state(w, 4)
    qkv, g, beta = I.round_stream(w, 1, 4)
    prev = I.previous_round(w, 4)
    n = np.array([9, -1, 3, 8], np.int32)
    dst, dcs, out, tdl, tk, status = run_fused(w, n, prev, qkv, cw, cs, g, beta, st)
    assert int(status.item()) & 0x1
    n_eff = np.where((n < 0) | (n > 8), 0, n).astype(np.int32)
    st1, cs1, _, ref = oracle_commit_then_verify(w, n_eff, prev, qkv, cw, cs, g, beta, st)
    assert torch.equal(dst[:, :2].cpu(), st[:, :2])
    assert_close(f64(dst), st1, "state")
    assert np.array_equal(f64(dcs), cs1)
    assert_close(f64(out), ref["out"], "out", bf16=True)


@pytest.mark.parametrize("D,Hk,Hv", [(128, 2, 4), (128, 2, 2), (64, 2, 4)])
def test_fused_round_loop_matches_oracle(gdnlib, D, Hk, Hv):
    """step_fused over three rounds plus flush against the oracle's verify / accept / rollback
    chain; the state carried on both sides."""
    w = small(I.WORKLOADS[2], L=3, B=6, N=8, Hk=Hk, Hv=Hv, D=D, V=2048, name="fusedloop%d_%d" % (D, Hv))
    cw, (st, cs) = I.model_weights(w), I.initial_state(w)
    dcw, dst, dcs = to_dev(cw, st, cs)
    r = SpecRound(w)
    d = oracle_dims(w)
    st_ref, cs_ref = f64(st), f64(cs)
    keep = []
    for rnd in range(3):
        qkv, g, beta = I.round_stream(w, rnd)
        lg, dr, _ = I.greedy_logits(w, rnd)
        dq, dg, db, dlg, ddr = to_dev(qkv, g, beta, lg, dr)
        keep.append((dq, dg))                     # the previous round's qkv / g stay alive
        r.step_fused(dq, dg, db, dlg, ddr, dcw, dst, dcs, round_=rnd)
        r.check_status()
        ref = oracle.verify(d, f64(qkv), f64(cw), cs_ref, f64(g), f64(beta), st_ref)
        n, _, _ = oracle.accept_greedy(logits_f32(lg), dr.numpy())
        assert np.array_equal(r.n_acc.cpu().numpy(), n)
        assert_close(f64(r.out), ref["out"], "out round %d" % rnd, bf16=True)
        assert_close(f64(r.tape_delta), ref["tape_delta"], "tape_delta round %d" % rnd)
        st_ref, cs_ref, _ = oracle.rollback(d, n, ref["tape_delta"], ref["tape_k"], f64(g),
                                            f64(qkv), st_ref, cs_ref)
    r.flush(dst, dcs)
    r.check_status()
    assert_close(f64(dst), st_ref, "state after flush")
    assert np.array_equal(f64(dcs), cs_ref)


def test_rollback_verify_full_size_sampled_units(gdnlib):
    """The bench workload's shape (30 layers, batch 64, N = 8), inputs drawn on the device; 16
    random (layer, sequence) units compared."""
    w = I.WORKLOADS[2]
    dev = "cuda"
    cw = I.model_weights(w, 0, dev)
    st, cs = I.initial_state(w, 0, dev)
    qkv, g, beta = I.round_stream(w, 1, 0, dev)
    prev = I.previous_round(w, 0, dev)
    n = prev[0]
    st0, cs0 = st.clone(), cs.clone()
    sh = _lib.GdnShape(L=w.L, B=w.B, T=w.N, Hk=w.Hk, Hv=w.Hv, Dk=w.D, Dv=w.D, W=w.W,
                       io_dtype=w.io_dtype)
    out = torch.empty(sh.out_shape(), dtype=w.io_dtype, device=dev)
    tdl = torch.empty(sh.out_shape(), dtype=torch.float32, device=dev)
    tk = torch.empty(sh.tape_k_shape(), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _lib.rollback_verify(sh, n, prev[1], prev[2], prev[3], prev[4], qkv, cw, cs, g, beta, st, out,
                         tdl, tk, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rng = np.random.default_rng(11)
    units = {(int(rng.integers(0, w.L)), int(rng.integers(0, w.B))) for _ in range(16)}
    nh = n.cpu().numpy()
    for (l, b) in sorted(units):
        sl = lambda t: t[l:l + 1, b:b + 1].cpu()
        prev_u = (None, sl(prev[1]), sl(prev[2]), sl(prev[3]), sl(prev[4]))
        st1, cs1, bad, ref = oracle_commit_then_verify(w, nh[b:b + 1], prev_u, sl(qkv),
                                                       cw[l:l + 1].cpu(), sl(cs0), sl(g), sl(beta),
                                                       sl(st0), L=1, B=1)
        assert bad == 0
        tag = "(l=%d,b=%d,n=%d)" % (l, b, nh[b])
        assert_close(f64(st[l:l + 1, b:b + 1]), st1, "state " + tag)
        assert np.array_equal(f64(cs[l:l + 1, b:b + 1]), cs1), "conv state " + tag
        assert_close(f64(out[l:l + 1, b:b + 1]), ref["out"], "out " + tag, bf16=True)
        assert_close(f64(tdl[l:l + 1, b:b + 1]), ref["tape_delta"], "delta " + tag)
