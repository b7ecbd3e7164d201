"""Pins of the CPU oracle against facts fixed outside the oracle itself: the pages' printed
values, closed forms, textbook special cases, independent formulations (numpy matrix forms,
brute force) and published known-answer vectors. CPU only."""
import os

import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import OracleDims

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------------------ helpers
def rand_inputs(rng, L=1, B=1, T=4, Hk=2, Hv=4, D=8, W=4, state_std=0.1):
    dims = OracleDims(L=L, B=B, T=T, Hk=Hk, Hv=Hv, Dk=D, Dv=D, W=W)
    C = dims.C
    x = dict(
        qkv=rng.standard_normal((L, B, T, C)),
        conv_w=rng.standard_normal((L, C, W)) * 0.5,
        conv_state=rng.standard_normal((L, B, W - 1, C)),
        g=np.exp(-np.logaddexp(0.0, rng.standard_normal((L, B, T, Hv)))),
        beta=1.0 / (1.0 + np.exp(-rng.standard_normal((L, B, T, Hv)))),
        state=rng.standard_normal((L, B, Hv, D, D)) * state_std,
    )
    return dims, x


def S_of(state):
    """Stored state [..., Dv, Dk] is S itself (row i in Dv, column j in Dk)."""
    return state


def silu(y):
    return y / (1.0 + np.exp(-y))


# ------------------------------------------------------------------------------ randomness
def test_philox_known_answer_vectors():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        v = [int(t, 16) for t in r]
        out = oracle.philox4x32_10(v[0:4], v[4:6])
        assert [int(o) for o in out] == v[6:10]


def test_draw_power_of_two_takes_top_bits():
    # floor(U * 2^k / 2^128) is the top k bits of the 128-bit output (x3 most significant)
    for ctr in range(20):
        x = oracle.philox4x32_10([ctr, 7, 3, 1], [0x1234, 0x5678])
        seed = 0x5678 << 32 | 0x1234
        for k in (1, 5, 17, 32):
            assert oracle.draw(seed, ctr, 7, 3, 1, 1 << k) == int(x[3]) >> (32 - k)
        top64 = int(x[3]) << 32 | int(x[2])
        for k in (33, 40, 60):
            assert oracle.draw(seed, ctr, 7, 3, 1, 1 << k) == top64 >> (64 - k)


def test_draw_is_uniform_below_Z():
    Z = 7
    r = np.array([oracle.draw(11, i, 0, 0, 0, Z) for i in range(70000)])
    assert r.min() >= 0 and r.max() < Z
    counts = np.bincount(r, minlength=Z)
    assert stats.chisquare(counts).pvalue > 1e-3


# ------------------------------------------------------------------------------ weights
def test_exp2_spec_error_bound_and_exact_points():
    rng = np.random.default_rng(0)
    x = -np.abs(rng.standard_normal(20000).astype(np.float32) * 12)
    e = oracle.exp2_spec(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(e - ref) / ref
    assert rel.max() < 2.0 ** -20
    ints = -np.arange(0, 65, dtype=np.float32)
    assert np.array_equal(oracle.exp2_spec(ints), np.exp2(ints))      # f = 0: exact powers
    assert oracle.exp2_spec(np.float32(0.0)) == 1.0
    assert np.all(oracle.exp2_spec(np.array([-64.6, -70, -1e4], np.float32)) == 0.0)


def test_scale_constant():
    for T in (0.7, 1.0, 0.25, 3.0):
        c = float(oracle.scale_c(T))
        # c = log2(e)/T rounded to fp32
        assert abs(c * float(np.float32(T)) * np.log(2.0) - 1.0) < 2 ** -23


def test_weights_track_softmax():
    rng = np.random.default_rng(1)
    row = (rng.standard_normal(500) * 2).astype(np.float32)
    T = 0.7
    w, Z = oracle.weights(row, T)
    m = row.max()
    assert w[np.argmax(row)] == 2 ** 32
    assert Z == int(w.sum())
    p = np.exp((row.astype(np.float64) - m) / np.float64(np.float32(T)))
    # fp32 exponent argument (|x| <= 64, relative error ~2^-23) and the floor to an integer
    assert np.allclose(w / 2.0 ** 32, p, rtol=1e-5, atol=2.0 ** -32)
    wb, Zb = oracle.weights(row, T, ban=3)
    assert wb[3] == 0 and Zb == Z - int(w[3])


# ------------------------------------------------------------------------------ greedy accept
def test_greedy_handcrafted_cases():
    V = 6
    lg = np.zeros((1, 4, V), np.float32)
    lg[0, 0, 2] = 5          # argmax row0 = 2
    lg[0, 1, 4] = 5          # argmax row1 = 4
    lg[0, 2, [1, 3]] = 5     # tie: lowest index 1
    lg[0, 3, 0] = 1          # bonus argmax 0
    n, out, bad = oracle.accept_greedy(lg, [[2, 4, 1]])
    assert bad == 0 and n[0] == 3 and list(out[0]) == [2, 4, 1, 0]
    n, out, _ = oracle.accept_greedy(lg, [[2, 4, 3]])   # 3 ties with 1 but is not the lowest
    assert n[0] == 2 and list(out[0]) == [2, 4, 1, -1]
    n, out, _ = oracle.accept_greedy(lg, [[0, 4, 1]])
    assert n[0] == 0 and list(out[0]) == [2, -1, -1, -1]
    n, out, bad = oracle.accept_greedy(lg, [[2, 9, 1]])  # token outside [0, V)
    assert bad == 4 and n[0] == 0 and list(out[0]) == [-1] * 4


def test_greedy_recovers_planted_lengths():
    import torch
    from speculative_verify_gdn_gb300 import inputs as I
    w0 = I.WORKLOADS[0]
    wb = I.custom(I.WORKLOADS[2], name="planted_bf16", L=1, B=64, N=8, V=4096, Hk=2, Hv=4, D=32)
    for w in (w0, wb):
        for rnd in range(6):
            lg, dr, L = I.greedy_logits(w, rnd)
            n, out, bad = oracle.accept_greedy(lg.float().numpy(), dr.numpy())
            assert bad == 0
            assert np.array_equal(n, L.numpy())
            am = lg.float().argmax(dim=2).numpy()
            for b in range(w.B):
                assert out[b, n[b]] == am[b, n[b]]
    del torch


def test_greedy_speculative_output_equals_plain_greedy():
    """xserv docs/25 §2: with a strict accept rule the output equals plain target greedy."""
    rng = np.random.default_rng(5)
    V, ctx = 40, 3
    table = rng.standard_normal((V, V, V)).astype(np.float32)   # next-token logits by last 2

    def target_logits(seq):
        return table[seq[-2], seq[-1]]

    def greedy_next(seq):
        return int(np.argmax(target_logits(seq)))

    seq0 = list(rng.integers(0, V, ctx))
    plain = list(seq0)
    while len(plain) < ctx + 60:
        plain.append(greedy_next(plain))
    spec = list(seq0)
    N = 4
    while len(spec) < ctx + 60:
        drafts, s = [], list(spec)
        for _ in range(N):     # a drafter that is right about 60% of the time
            t = greedy_next(s) if rng.random() < 0.6 else int(rng.integers(0, V))
            drafts.append(t)
            s.append(t)
        rows = np.stack([target_logits(spec + drafts[:i]) for i in range(N + 1)])[None]
        n, out, _ = oracle.accept_greedy(rows, [drafts])
        spec += [int(t) for t in out[0, : n[0] + 1]]
    assert spec[: ctx + 60] == plain


# ------------------------------------------------------------------------------ sampling accept
def softmax64(row, T):
    z = row.astype(np.float64) / np.float64(np.float32(T))
    z -= z.max()
    e = np.exp(z)
    return e / e.sum()


def chisq_p(counts, probs):
    n = counts.sum()
    exp = probs * n
    keep = exp >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    ex = np.append(exp[keep], exp[~keep].sum())
    if ex[-1] == 0:
        obs, ex = obs[:-1], ex[:-1]
    return stats.chisquare(obs, ex * obs.sum() / ex.sum()).pvalue


@pytest.mark.slow
def test_sampling_first_token_follows_target_distribution():
    """colibrì ch.08 §5: with accept-with-p(draft) and ban+renormalise, the emitted token is
    distributed exactly as p (10^6 draws, chi-square)."""
    rng = np.random.default_rng(7)
    V, T = 48, 0.7
    lg = (rng.standard_normal((1, 2, V)) * 2).astype(np.float32)
    p0 = softmax64(lg[0, 0], T)
    Bn = 1_000_000
    for drafts in (np.full((Bn, 1), int(np.argsort(p0)[-3])),       # fixed draft
                   rng.integers(0, V, (Bn, 1))):                     # varied drafts
        n, out, bad = oracle.accept_sample(lg, drafts, T, seed=123, round_=9, seq_shared=True,
                                           B=Bn)
        assert bad == 0
        counts = np.bincount(out[:, 0], minlength=V)
        assert chisq_p(counts, p0) > 1e-3
        # rejection never re-emits the banned draft
        rej = n == 0
        assert not np.any(out[rej, 0] == drafts[rej, 0])


@pytest.mark.slow
def test_sampling_bonus_follows_last_row():
    rng = np.random.default_rng(8)
    V, T = 32, 1.3
    lg = (rng.standard_normal((1, 3, V)) * 2).astype(np.float32)
    d = np.array([3, 5])
    lg[0, 0, 3] = 200.0
    lg[0, 1, 5] = 200.0       # p(draft) = 1 in both draft rows
    Bn = 400_000
    n, out, _ = oracle.accept_sample(lg, np.tile(d, (Bn, 1)), T, 5, 1, seq_shared=True, B=Bn)
    assert np.all(n == 2)
    assert chisq_p(np.bincount(out[:, 2], minlength=V), softmax64(lg[0, 2], T)) > 1e-3


def test_sampling_point_probabilities():
    rng = np.random.default_rng(9)
    V, T = 20, 0.7
    lg = (rng.standard_normal((1, 4, V))).astype(np.float32)
    lg[0, 0, 7] = -1000.0          # p(7) = 0 in row 0: always rejected, never emitted
    Bn = 20000
    n, out, _ = oracle.accept_sample(lg, np.tile([7, 1, 2], (Bn, 1)), T, 1, 2, seq_shared=True,
                                     B=Bn)
    assert np.all(n == 0) and not np.any(out[:, 0] == 7)
    # P(all N accepted) = prod_i p_i(d_i)
    d = [int(np.argmax(lg[0, i])) for i in range(3)]
    lg2 = lg.copy()
    lg2[0, 0, 7] = 0.0
    d = [int(np.argmax(lg2[0, i])) for i in range(3)]
    pall = np.prod([softmax64(lg2[0, i], T)[d[i]] for i in range(3)])
    n, _, _ = oracle.accept_sample(lg2, np.tile(d, (Bn * 5, 1)), T, 3, 4, seq_shared=True,
                                   B=Bn * 5)
    k = int((n == 3).sum())
    sd = np.sqrt(Bn * 5 * pall * (1 - pall))
    assert abs(k - Bn * 5 * pall) < 5 * sd


def test_sampling_greedy_at_zero_temperature():
    rng = np.random.default_rng(10)
    lg = rng.standard_normal((3, 5, 50)).astype(np.float32)
    dr = rng.integers(0, 50, (3, 4))
    a = oracle.accept_sample(lg, dr, 0.0, 1, 1)
    b = oracle.accept_greedy(lg, dr)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ------------------------------------------------------------------------------ conv + norm
def test_conv_matches_numpy_correlate():
    rng = np.random.default_rng(11)
    dims, x = rand_inputs(rng, T=5, Hk=1, Hv=2, D=4, W=4)
    # S_0 = 0, g = 1, beta = 1: delta_0 = v_0 exposes the conv output of the v channels
    x["state"][:] = 0.0
    x["g"][:] = 1.0
    x["beta"][:] = 1.0
    r = oracle.verify(dims, **x)
    C, W = dims.C, dims.W
    y = np.zeros((dims.T, C))
    for c in range(C):
        xh = np.concatenate([x["conv_state"][0, 0, :, c], x["qkv"][0, 0, :, c]])
        y[:, c] = silu(np.correlate(xh, x["conv_w"][0, c], mode="valid"))
    Dk = dims.Dk
    k = y[:, Dk:2 * Dk]
    k = k / np.sqrt((k * k).sum(1, keepdims=True) + dims.l2_eps)
    assert np.allclose(r["tape_k"][0, 0, :, 0], k, rtol=1e-12, atol=1e-14)
    v0 = y[0, 2 * Dk:]
    assert np.allclose(r["tape_delta"][0, 0, 0].ravel(), v0, rtol=1e-12, atol=1e-14)


def test_conv_impulse_returns_taps():
    dims = OracleDims(L=1, B=1, T=4, Hk=1, Hv=1, Dk=4, Dv=4, W=4, act_silu=False)
    rng = np.random.default_rng(12)
    C = dims.C
    qkv = np.zeros((1, 1, 4, C))
    c = 2 * 4 + 1          # a v channel
    qkv[0, 0, 0, c] = 1.0
    w = rng.standard_normal((1, C, 4))
    x = dict(qkv=qkv, conv_w=w, conv_state=np.zeros((1, 1, 3, C)), g=np.ones((1, 1, 4, 1)),
             beta=np.ones((1, 1, 4, 1)), state=np.zeros((1, 1, 1, 4, 4)))
    r = oracle.verify(dims, **x)
    # delta_t = v_t - g S_{t-1} k_t; with zero keys (k = 0 after norm of 0) delta_t = v_t = w[W-1-t]
    got = r["tape_delta"][0, 0, :, 0, 1]
    assert np.allclose(got, w[0, c, ::-1], rtol=0, atol=1e-15)


def test_literal_mode_is_plain_normalisation():
    # W = 1, taps 1, no activation: q, k are the raw rows L2-normalised (the tiny workload's text)
    rng = np.random.default_rng(13)
    dims = OracleDims(L=1, B=2, T=3, Hk=2, Hv=2, Dk=8, Dv=8, W=1, act_silu=False)
    C = dims.C
    qkv = rng.standard_normal((1, 2, 3, C))
    x = dict(qkv=qkv, conv_w=np.ones((1, C, 1)), conv_state=np.zeros((1, 2, 0, C)),
             g=np.full((1, 2, 3, 2), 0.9), beta=np.full((1, 2, 3, 2), 0.5),
             state=rng.standard_normal((1, 2, 2, 8, 8)))
    r = oracle.verify(dims, **x)
    k = qkv[..., 16:32].reshape(1, 2, 3, 2, 8)
    k = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
    assert np.allclose(r["tape_k"], k, rtol=1e-13, atol=0)
    assert np.allclose(np.linalg.norm(r["tape_k"], axis=-1), 1.0, atol=1e-6)


# ------------------------------------------------------------------------------ recurrence
def literal(rng, T, Hk, Hv, D, B=1, g=None, beta=None, state=None, l2_eps=0.0, qkv=None):
    dims = OracleDims(L=1, B=B, T=T, Hk=Hk, Hv=Hv, Dk=D, Dv=D, W=1, act_silu=False,
                      l2_eps=l2_eps)
    C = dims.C
    x = dict(qkv=rng.standard_normal((1, B, T, C)) if qkv is None else qkv,
             conv_w=np.ones((1, C, 1)), conv_state=np.zeros((1, B, 0, C)),
             g=rng.uniform(0.2, 1.0, (1, B, T, Hv)) if g is None else g,
             beta=rng.uniform(0.0, 1.0, (1, B, T, Hv)) if beta is None else beta,
             state=rng.standard_normal((1, B, Hv, D, D)) * 0.3 if state is None else state)
    return dims, x


def split_qkv(dims, qkv):
    Hk, Hv, D = dims.Hk, dims.Hv, dims.Dk
    q = qkv[..., :Hk * D].reshape(*qkv.shape[:-1], Hk, D)
    k = qkv[..., Hk * D:2 * Hk * D].reshape(*qkv.shape[:-1], Hk, D)
    v = qkv[..., 2 * Hk * D:].reshape(*qkv.shape[:-1], Hv, D)
    nq = q / np.sqrt((q * q).sum(-1, keepdims=True) + dims.l2_eps)
    nk = k / np.sqrt((k * k).sum(-1, keepdims=True) + dims.l2_eps)
    return nq, nk, v


def test_beta_zero_is_pure_decay():
    rng = np.random.default_rng(20)
    dims, x = literal(rng, T=5, Hk=1, Hv=2, D=6, beta=np.zeros((1, 1, 5, 2)))
    r = oracle.verify(dims, node_states=True, **x)
    S0 = S_of(x["state"][0, 0])
    G = np.cumprod(x["g"][0, 0], axis=0)     # [T, Hv]
    for t in range(5):
        assert np.allclose(S_of(r["node_state"][0, 0, t]), G[t][:, None, None] * S0, rtol=1e-13)
    assert np.allclose(r["tape_delta"], 0.0)


def test_beta_one_writes_value():
    # delta rule with ||k|| = 1, beta = 1: S_t k_t = v_t exactly (the key is overwritten)
    rng = np.random.default_rng(21)
    dims, x = literal(rng, T=6, Hk=2, Hv=4, D=8, beta=np.ones((1, 1, 6, 4)))
    r = oracle.verify(dims, node_states=True, **x)
    _, k, v = split_qkv(dims, x["qkv"][0, 0])
    for t in range(6):
        for h in range(4):
            St = S_of(r["node_state"][0, 0, t, h])
            assert np.allclose(St @ k[t, h // 2], v[t, h], rtol=1e-12, atol=1e-12)


def test_linear_associative_memory():
    # g = 1, beta = 1, S_0 = 0, orthonormal keys: S = sum_t v_t k_t^T (textbook outer-product memory)
    rng = np.random.default_rng(22)
    D, T = 8, 5
    dims = OracleDims(L=1, B=1, T=T, Hk=1, Hv=1, Dk=D, Dv=D, W=1, act_silu=False, l2_eps=0.0)
    Q, _ = np.linalg.qr(rng.standard_normal((D, D)))
    qkv = np.zeros((1, 1, T, dims.C))
    qkv[0, 0, :, :D] = rng.standard_normal((T, D))
    qkv[0, 0, :, D:2 * D] = Q[:T] * 3.0
    qkv[0, 0, :, 2 * D:] = rng.standard_normal((T, D))
    _, x = literal(rng, T, 1, 1, D, g=np.ones((1, 1, T, 1)), beta=np.ones((1, 1, T, 1)),
                   state=np.zeros((1, 1, 1, D, D)), qkv=qkv)
    r = oracle.verify(dims, node_states=True, **x)
    mem = sum(np.outer(qkv[0, 0, t, 2 * D:], Q[t]) for t in range(T))
    assert np.allclose(S_of(r["node_state"][0, 0, T - 1, 0]), mem, atol=1e-12)
    q = qkv[0, 0, :, :D] / np.linalg.norm(qkv[0, 0, :, :D], axis=1, keepdims=True)
    assert np.allclose(r["out"][0, 0, :, 0], np.einsum("tij,tj->ti",
                       np.stack([S_of(r["node_state"][0, 0, t, 0]) for t in range(T)]), q),
                       atol=1e-12)


def test_matrix_form_of_the_delta_rule():
    """S_t = g_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = scale * S_t q_t,
    evaluated independently with numpy matrices."""
    rng = np.random.default_rng(23)
    for Hk, Hv in ((1, 1), (2, 4)):
        dims, x = literal(rng, T=7, Hk=Hk, Hv=Hv, D=6, B=2, l2_eps=1e-6)
        dims.qk_scale = 0.37
        r = oracle.verify(dims, node_states=True, **x)
        for b in range(2):
            q, k, v = split_qkv(dims, x["qkv"][0, b])
            for h in range(Hv):
                S = S_of(x["state"][0, b, h]).copy()
                kh = h // (Hv // Hk)
                for t in range(7):
                    gt, bt = x["g"][0, b, t, h], x["beta"][0, b, t, h]
                    kk = k[t, kh]
                    S = gt * S @ (np.eye(6) - bt * np.outer(kk, kk)) + bt * np.outer(v[t, h], kk)
                    assert np.allclose(S_of(r["node_state"][0, b, t, h]), S, rtol=1e-12,
                                       atol=1e-13)
                    assert np.allclose(r["out"][0, b, t, h], 0.37 * S @ q[t, kh], rtol=1e-12,
                                       atol=1e-13)


# ------------------------------------------------------------------------------ rollback
def test_rollback_equals_sequential_run_bit_identical():
    """GDN investigation §4: restore + replay of the n accepted steps = the sequential run over
    only the committed tokens. Both apply the same expression in the same order: bit-identical."""
    rng = np.random.default_rng(30)
    dims, x = rand_inputs(rng, L=2, B=3, T=6, Hk=2, Hv=4, D=6)
    full = oracle.verify(dims, **x)
    n_acc = np.array([0, 3, 6], np.int32)
    st, cs, bad = oracle.rollback(dims, n_acc, full["tape_delta"], full["tape_k"], x["g"],
                                  x["qkv"], x["state"], x["conv_state"])
    assert bad == 0
    for b, n in enumerate(n_acc):
        if n == 0:
            assert np.array_equal(st[:, b], x["state"][:, b])
            assert np.array_equal(cs[:, b], x["conv_state"][:, b])
            continue
        sub = OracleDims(L=2, B=1, T=int(n), Hk=2, Hv=4, Dk=6, Dv=6, W=4)
        xs = {k: v[:, b:b + 1, :n] if k in ("qkv", "g", "beta") else v[:, b:b + 1]
              for k, v in x.items() if k != "conv_w"}
        seq = oracle.verify(sub, conv_w=x["conv_w"], node_states=True, **xs)
        assert np.array_equal(st[:, b], seq["node_state"][:, 0, n - 1])
        xh = np.concatenate([x["conv_state"][:, b], x["qkv"][:, b, :n]], axis=1)
        assert np.array_equal(cs[:, b], xh[:, -3:])


def test_rollback_rejects_out_of_range_counts():
    rng = np.random.default_rng(31)
    dims, x = rand_inputs(rng, B=2, T=3)
    full = oracle.verify(dims, **x)
    st, cs, bad = oracle.rollback(dims, np.array([4, -1], np.int32), full["tape_delta"],
                                  full["tape_k"], x["g"], x["qkv"], x["state"], x["conv_state"])
    assert bad == 1 and np.array_equal(st, x["state"])


# ------------------------------------------------------------------------------ tree
def tree_parents(rng, T, depth, branch):
    par = [-1]
    dep = [1]
    kids = {-1: 1}
    for v in range(1, T):
        if v < depth:
            p = v - 1
        else:
            cand = [u for u in range(-1, v) if (u < 0 or dep[u] < depth) and kids.get(u, 0) < branch]
            p = int(rng.choice(cand))
        par.append(p)
        dep.append(1 if p < 0 else dep[p] + 1)
        kids[p] = kids.get(p, 0) + 1
    return np.array(par, np.int32)


def test_tree_matches_chain_along_every_path():
    rng = np.random.default_rng(40)
    T = 12
    dims, x = rand_inputs(rng, L=1, B=2, T=T, Hk=1, Hv=2, D=5)
    par = np.stack([tree_parents(rng, T, 5, 3), tree_parents(rng, T, 5, 3)])
    tr = oracle.verify(dims, parent=par, node_states=True, **x)
    for b in range(2):
        for leaf in [v for v in range(T) if v not in par[b]]:
            path, u = [], leaf
            while u >= 0:
                path.append(u)
                u = par[b, u]
            path.reverse()
            n = len(path)
            sub = OracleDims(L=1, B=1, T=n, Hk=1, Hv=2, Dk=5, Dv=5, W=4)
            xs = dict(qkv=x["qkv"][:, b:b + 1, path], g=x["g"][:, b:b + 1, path],
                      beta=x["beta"][:, b:b + 1, path], conv_state=x["conv_state"][:, b:b + 1],
                      state=x["state"][:, b:b + 1], conv_w=x["conv_w"])
            ch = oracle.verify(sub, node_states=True, **xs)
            assert np.array_equal(tr["out"][:, b, path], ch["out"][:, 0])
            assert np.array_equal(tr["tape_delta"][:, b, path], ch["tape_delta"][:, 0])
            assert np.array_equal(tr["node_state"][:, b, path], ch["node_state"][:, 0])


def root_to_leaf(par_b, leaf):
    path, u = [], int(leaf)
    while u >= 0:
        path.append(u)
        u = int(par_b[u])
    return path[::-1]


@pytest.mark.parametrize("gate_dk", [False, True])
def test_path_rollback_equals_chain_over_the_path(gate_dk):
    """GDN investigation §4 tape replay along an accepted tree path (§2.2 tree verification):
    restoring the snapshot and replaying the tape of nodes path[0..n-1] equals the sequential
    recurrence run over only those nodes' rows, bit for bit (the same expression in the same
    order), and equals the tree verify's own state of node path[n-1]; the conv state becomes the
    last W-1 rows of conv_state ++ qkv[path[:n]] (the path nodes' raw rows, not rows 0..n-1)."""
    rng = np.random.default_rng(60 + int(gate_dk))
    T, L, B, Hk, Hv, D, W, depth = 13, 2, 3, 1, 2, 5, 4, 6
    dims, x = rand_inputs(rng, L=L, B=B, T=T, Hk=Hk, Hv=Hv, D=D, W=W)
    if gate_dk:
        x["g"] = np.exp(-np.logaddexp(0.0, rng.standard_normal((L, B, T, Hv, D))))
    par = np.stack([tree_parents(rng, T, depth, 3) for _ in range(B)])
    tr = oracle.verify(dims, parent=par, node_states=True, **x)
    # each sequence accepts a path to a random leaf that is not the creation-order chain 0,1,2..
    paths = []
    for b in range(B):
        leaves = [v for v in range(T) if v not in par[b]]
        cand = [lf for lf in leaves if root_to_leaf(par[b], lf) != list(range(len(root_to_leaf(par[b], lf))))]
        paths.append(root_to_leaf(par[b], rng.choice(cand if cand else leaves)))
    assert any(p != list(range(len(p))) for p in paths)
    P = depth
    pth = np.full((B, P), -1, np.int32)
    for b, p in enumerate(paths):
        pth[b, :len(p)] = p
    cuts = [sorted({0, 1, len(p) - 1, len(p)}) for p in paths]
    for k in range(4):
        n_acc = np.array([c[min(k, len(c) - 1)] for c in cuts], np.int32)
        st, cs, bad = oracle.rollback(dims, n_acc, tr["tape_delta"], tr["tape_k"], x["g"],
                                      x["qkv"], x["state"], x["conv_state"], path=pth)
        assert bad == 0
        for b, n in enumerate(n_acc):
            n = int(n)
            if n == 0:
                assert np.array_equal(st[:, b], x["state"][:, b])
                assert np.array_equal(cs[:, b], x["conv_state"][:, b])
                continue
            nodes = paths[b][:n]
            # the tree verify's state of the last accepted node
            assert np.array_equal(st[:, b], tr["node_state"][:, b, nodes[-1]])
            # the chain recurrence over only the path nodes' rows
            sub = OracleDims(L=L, B=1, T=n, Hk=Hk, Hv=Hv, Dk=D, Dv=D, W=W)
            xs = dict(qkv=x["qkv"][:, b:b + 1, nodes], g=x["g"][:, b:b + 1, nodes],
                      beta=x["beta"][:, b:b + 1, nodes], conv_state=x["conv_state"][:, b:b + 1],
                      state=x["state"][:, b:b + 1], conv_w=x["conv_w"])
            ch = oracle.verify(sub, node_states=True, **xs)
            assert np.array_equal(st[:, b], ch["node_state"][:, 0, n - 1])
            xh = np.concatenate([x["conv_state"][:, b], x["qkv"][:, b, nodes]], axis=1)
            assert np.array_equal(cs[:, b], xh[:, -(W - 1):])


def test_path_rollback_rejects_bad_nodes_and_counts():
    """A path node outside [0, T) sets bit 8, a count beyond the path capacity bit 1; either
    leaves that sequence's state and conv state untouched while the others commit."""
    rng = np.random.default_rng(62)
    T, depth = 8, 4
    dims, x = rand_inputs(rng, L=1, B=3, T=T, Hk=1, Hv=2, D=4)
    par = np.stack([tree_parents(rng, T, depth, 3) for _ in range(3)])
    tr = oracle.verify(dims, parent=par, **x)
    pth = np.full((3, depth), -1, np.int32)
    for b in range(3):
        p = root_to_leaf(par[b], [v for v in range(T) if v not in par[b]][0])
        pth[b, :len(p)] = p
    pth[0, 1] = T                     # out of range node
    n_acc = np.array([2, 1, depth + 1], np.int32)
    st, cs, bad = oracle.rollback(dims, n_acc, tr["tape_delta"], tr["tape_k"], x["g"], x["qkv"],
                                  x["state"], x["conv_state"], path=pth)
    assert bad == (8 | 1)
    for b in (0, 2):
        assert np.array_equal(st[:, b], x["state"][:, b])
        assert np.array_equal(cs[:, b], x["conv_state"][:, b])
    assert not np.array_equal(st[:, 1], x["state"][:, 1])
    pth[0, 1] = -2                    # negative node
    st, cs, bad = oracle.rollback(dims, np.array([2, 0, 0], np.int32), tr["tape_delta"],
                                  tr["tape_k"], x["g"], x["qkv"], x["state"], x["conv_state"],
                                  path=pth)
    assert bad == 8 and np.array_equal(st, x["state"]) and np.array_equal(cs, x["conv_state"])


def test_chain_shaped_tree_equals_chain():
    rng = np.random.default_rng(41)
    dims, x = rand_inputs(rng, L=1, B=2, T=5)
    par = np.tile(np.arange(-1, 4, dtype=np.int32), (2, 1))
    a = oracle.verify(dims, parent=par, **x)
    b = oracle.verify(dims, **x)
    for k in a:
        assert np.array_equal(a[k], b[k])


def test_tree_accept_matches_brute_force():
    rng = np.random.default_rng(42)
    T, V, P = 14, 6, 5
    for trial in range(200):
        par = tree_parents(rng, T, 5, 3)
        tok = rng.integers(0, V, T).astype(np.int32)
        lg = rng.standard_normal((1, T + 1, V)).astype(np.float32)
        path, n, out, bad = oracle.accept_tree(lg, par[None], tok[None], P)
        assert bad == 0
        am = lg[0].argmax(1)
        # brute force: v is matched iff its parent is matched (or is the context) and its token is
        # the argmax of the parent's row; keep the lowest-numbered matched child at each step
        matched_child = {}
        for v in range(T):
            p = par[v]
            if tok[v] == am[0 if p < 0 else 1 + p] and p not in matched_child:
                matched_child[p] = v
        chain, cur = [], -1
        while cur in matched_child and len(chain) < P:
            cur = matched_child[cur]
            chain.append(cur)
        assert n[0] == len(chain)
        assert list(path[0, :n[0]]) == chain
        last = -1 if not chain else chain[-1]
        assert list(out[0, :n[0] + 1]) == [int(tok[c]) for c in chain] + [int(am[1 + last])]


# ------------------------------------------------------------------------------ workload generator
def test_all_accepted_probability_matches_printed_values():
    import torch
    from speculative_verify_gdn_gb300 import inputs as I
    rows = [ln.split()[:3] for ln in open(os.path.join(GOLDEN, "all_accept_probabilities.txt"))
            if ln.strip() and not ln.startswith("#")]
    for a, N, printed in rows:
        a, N, printed = float(a), int(N), float(printed) / 100
        # the printed numbers are alpha^N, rounded as the pages print them
        assert abs(a ** N - printed) <= 0.5 * 10 ** -(len(str(printed).split(".")[-1])) + 1e-12 \
            or abs(a ** N / printed - 1) < 0.03
        w = I.custom(I.WORKLOADS[2], name="gen_%g_%d" % (a, N), B=200000, N=N, alphas=(a,))
        L = I.accept_lengths(w, 0)
        frac = float((L == N).double().mean())
        sd = np.sqrt(a ** N * (1 - a ** N) / w.B)
        assert abs(frac - a ** N) < 5 * sd
    del torch


# ------------------------------------------------------------------------------ NaN logits
def test_nan_logits_count_as_negative_infinity():
    """The one NaN rule of both sides: a NaN logit is never the argmax (a row of NaN / −∞ gives
    index 0, like a tie) and has sampling weight 0."""
    nan, inf = np.float32("nan"), np.float32("inf")
    row = np.array([nan, 1.0, 3.0, nan, 3.0, -2.0], np.float32)
    assert oracle.argmax(row) == 2
    assert oracle.argmax(np.full(7, nan, np.float32)) == 0
    assert oracle.argmax(np.array([nan, -inf, nan, -inf], np.float32)) == 0
    assert oracle.argmax(np.array([nan, nan, -5.0, nan], np.float32)) == 2
    lg = np.stack([row, np.where(np.isnan(row), -inf, row)])[None]         # [1, 2, 6]
    # greedy: the NaN row behaves as the row with −∞ in place of each NaN
    n, out, _ = oracle.accept_greedy(lg, np.array([[2]], np.int32))
    assert n[0] == 1 and list(out[0]) == [2, 2]
    # sampling: the NaN positions are never drawn, and the two rows give the same draws
    for seed in range(200):
        a = oracle.accept_sample(lg[:, :1].repeat(2, 1), np.array([[1]], np.int32), 0.7, seed, 0)
        b = oracle.accept_sample(lg[:, 1:].repeat(2, 1), np.array([[1]], np.int32), 0.7, seed, 0)
        assert np.array_equal(a[1], b[1]) and a[0][0] == b[0][0]
        assert not np.isnan(row[a[1][0, 0]])


# ------------------------------------------------------------------------------ threads
def test_threaded_oracle_is_bit_identical_to_serial():
    """The oracle's thread count only splits independent units (layers x sequences, sequences)
    between threads: every output is bit-identical to the single-threaded run."""
    rng = np.random.default_rng(70)
    dims, x = rand_inputs(rng, L=3, B=5, T=6, Hk=2, Hv=4, D=8)
    par = np.stack([tree_parents(rng, 6, 4, 3) for _ in range(5)])
    V = 300
    lg = (rng.standard_normal((5, 7, V)) * 2).astype(np.float32)
    dr = lg[:, :6].argmax(-1).astype(np.int32)
    dr[::2, 1] = (dr[::2, 1] + 1) % V
    tok = rng.integers(0, V, (5, 6)).astype(np.int32)
    res = []
    for threads in (1, 4):
        oracle.set_threads(threads)
        try:
            v = oracle.verify(dims, **x)
            t = oracle.verify(dims, parent=par, node_states=True, **x)
            n = np.array([0, 6, 3, 1, 5], np.int32)
            r = oracle.rollback(dims, n, v["tape_delta"], v["tape_k"], x["g"], x["qkv"], x["state"],
                                x["conv_state"])
            a = oracle.accept_sample(lg, dr, 0.7, 9, 2)
            gr = oracle.accept_greedy(lg, dr)
            tr = oracle.accept_tree(lg, par, tok, 4)
        finally:
            oracle.set_threads(1)
        res.append([v["out"], v["tape_delta"], v["tape_k"], t["out"], t["node_state"], r[0], r[1],
                    a[0], a[1], gr[0], gr[1], tr[0], tr[1], tr[2]])
    for u, w in zip(*res):
        assert np.array_equal(u, w)
