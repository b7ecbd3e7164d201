"""The attention-layer oracle (the hybrid's full-attention verify over a KV cache and the cache
truncation on reject, GDN investigation §2.1 / §2.2) pinned to closed forms and invariants: one
visible key returns its value exactly (and shows the query-head -> kv-head mapping), equal keys
give the mean of the visible values (the causal count), orthogonal keys with one aligned query
give that key's value, and cache order, later positions, the append and truncation behave as the
definitions fix."""
import numpy as np
import pytest

import oracle
from oracle import AttnDims


def rand_attn(rng, L=1, B=2, T=4, Hq=4, Hkv=2, D=8, ctx=16, lens=(3, 7)):
    d = AttnDims(L=L, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, ctx=ctx)
    kv_len = np.array([lens[b % len(lens)] for b in range(B)], np.int32)
    q = rng.standard_normal((L, B, T, Hq, D))
    kn = rng.standard_normal((L, B, T, Hkv, D))
    vn = rng.standard_normal((L, B, T, Hkv, D))
    kc = np.zeros((L, B, Hkv, ctx, D))
    vc = np.zeros((L, B, Hkv, ctx, D))
    for b in range(B):
        kc[:, b, :, :kv_len[b]] = rng.standard_normal((L, Hkv, kv_len[b], D))
        vc[:, b, :, :kv_len[b]] = rng.standard_normal((L, Hkv, kv_len[b], D))
    return d, kv_len, q, kn, vn, kc, vc


def test_single_visible_key_returns_its_value_and_the_head_mapping():
    rng = np.random.default_rng(1)
    d, _, q, kn, vn, kc, vc = rand_attn(rng, B=1, T=1, Hq=6, Hkv=2, lens=(0,))
    out, _, _, bad = oracle.attn_verify(d, [0], q, kn, vn, kc, vc)
    assert bad == 0
    for hq in range(6):
        # softmax over one key is exactly 1: o = v of kv head hq // 3
        assert np.array_equal(out[0, 0, 0, hq], vn[0, 0, 0, hq // 3])


def test_equal_keys_average_the_visible_values():
    rng = np.random.default_rng(2)
    d, kv_len, q, kn, vn, kc, vc = rand_attn(rng, B=2, T=3, lens=(5, 0))
    kstar = rng.standard_normal(d.D)
    kn[:] = kstar
    for b in range(d.B):
        kc[:, b, :, :kv_len[b]] = kstar
    out, _, _, bad = oracle.attn_verify(d, kv_len, q, kn, vn, kc, vc)
    assert bad == 0
    for b in range(d.B):
        n0 = kv_len[b]
        for i in range(d.T):
            for hq in range(d.Hq):
                h = hq // (d.Hq // d.Hkv)
                rows = np.concatenate([vc[0, b, h, :n0], vn[0, b, :i + 1, h]], axis=0)
                assert rows.shape[0] == n0 + i + 1       # rows 0 .. n0+i are visible
                np.testing.assert_allclose(out[0, b, i, hq], rows.mean(axis=0), rtol=1e-12,
                                           atol=1e-13)


def test_aligned_query_selects_one_orthogonal_key():
    D, n0 = 16, 9
    rng = np.random.default_rng(3)
    d = AttnDims(L=1, B=1, T=1, Hq=1, Hkv=1, D=D, ctx=n0 + 1, scale=1.0)
    kc = np.zeros((1, 1, 1, n0 + 1, D))
    vc = np.zeros_like(kc)
    kc[0, 0, 0, :n0] = np.eye(D)[:n0]              # key j = e_j
    vc[0, 0, 0, :n0] = rng.standard_normal((n0, D))
    kn = np.zeros((1, 1, 1, 1, D))
    kn[..., n0] = 1.0                              # the new key e_n0
    vn = rng.standard_normal((1, 1, 1, 1, D))
    m, alpha = 4, 60.0
    q = np.zeros((1, 1, 1, 1, D))
    q[..., m] = alpha                              # scores: alpha for key m, 0 for the rest
    out, _, _, _ = oracle.attn_verify(d, [n0], q, kn, vn, kc, vc)
    # weight of key m is 1 / (1 + n0 e^-alpha); every other weight is e^-alpha / (1 + n0 e^-alpha)
    vmax = max(np.abs(vc).max(), np.abs(vn).max())
    assert np.abs(out[0, 0, 0, 0] - vc[0, 0, 0, m]).max() <= 2 * n0 * np.exp(-alpha) * vmax


def test_cache_order_is_irrelevant_and_later_positions_are_not_seen():
    rng = np.random.default_rng(4)
    d, kv_len, q, kn, vn, kc, vc = rand_attn(rng, L=2, B=2, T=4, lens=(6, 2))
    ref, _, _, _ = oracle.attn_verify(d, kv_len, q, kn, vn, kc, vc)
    kc2, vc2 = kc.copy(), vc.copy()
    for b in range(d.B):
        perm = rng.permutation(kv_len[b])
        kc2[:, b, :, :kv_len[b]] = np.take(kc[:, b], perm, axis=2)
        vc2[:, b, :, :kv_len[b]] = np.take(vc[:, b], perm, axis=2)
    out2, _, _, _ = oracle.attn_verify(d, kv_len, q, kn, vn, kc2, vc2)
    np.testing.assert_allclose(out2, ref, rtol=1e-12, atol=1e-13)
    # changing positions i >= 2 leaves rows 0, 1 bit-identical and changes row 2
    kn3, vn3 = kn.copy(), vn.copy()
    kn3[:, :, 2:] += 1.0
    vn3[:, :, 2:] -= 2.0
    out3, _, _, _ = oracle.attn_verify(d, kv_len, q, kn3, vn3, kc, vc)
    assert np.array_equal(out3[:, :, :2], ref[:, :, :2])
    assert not np.allclose(out3[:, :, 2], ref[:, :, 2])


def test_values_enter_linearly_and_scale_multiplies_the_scores():
    rng = np.random.default_rng(5)
    d, kv_len, q, kn, vn, kc, vc = rand_attn(rng)
    a, _, _, _ = oracle.attn_verify(d, kv_len, q, kn, vn, kc, vc)
    b2, _, _, _ = oracle.attn_verify(d, kv_len, q, kn, 2 * vn + 1, kc, 2 * vc + 1)
    # the softmax weights sum to 1, so an affine map of every value maps the output the same way
    np.testing.assert_allclose(b2, 2 * a + 1, rtol=1e-12, atol=1e-12)
    d2 = AttnDims(L=d.L, B=d.B, T=d.T, Hq=d.Hq, Hkv=d.Hkv, D=d.D, ctx=d.ctx, scale=0.37)
    d3 = AttnDims(L=d.L, B=d.B, T=d.T, Hq=d.Hq, Hkv=d.Hkv, D=d.D, ctx=d.ctx, scale=1.0)
    x, _, _, _ = oracle.attn_verify(d2, kv_len, q, kn, vn, kc, vc)
    y, _, _, _ = oracle.attn_verify(d3, kv_len, 0.37 * q, kn, vn, kc, vc)
    np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-13)


def test_append_writes_exactly_the_new_rows():
    rng = np.random.default_rng(6)
    d, kv_len, q, kn, vn, kc, vc = rand_attn(rng, L=2, B=2, T=3, ctx=12, lens=(4, 9))
    _, kc2, vc2, bad = oracle.attn_verify(d, kv_len, q, kn, vn, kc, vc)
    assert bad == 0
    for b in range(d.B):
        n0 = kv_len[b]
        for i in range(d.T):
            assert np.array_equal(kc2[:, b, :, n0 + i], kn[:, b, i])
            assert np.array_equal(vc2[:, b, :, n0 + i], vn[:, b, i])
        keep = np.ones(d.ctx, bool)
        keep[n0:n0 + d.T] = False
        assert np.array_equal(kc2[:, b, :, keep], kc[:, b, :, keep])
        assert np.array_equal(vc2[:, b, :, keep], vc[:, b, :, keep])


def test_length_out_of_range_is_reported_and_skipped():
    rng = np.random.default_rng(7)
    d, _, q, kn, vn, kc, vc = rand_attn(rng, B=2, T=4, ctx=10)
    out, kc2, _, bad = oracle.attn_verify(d, [7, 6], q, kn, vn, kc, vc)   # 7 + 4 > 10
    assert bad == 1
    assert not out[:, 0].any() and np.array_equal(kc2[:, 0], kc[:, 0])
    assert out[:, 1].any()


def test_truncate_worked_example():
    kl, bad = oracle.attn_truncate(4, [0, 4, 2, 5, -1], [10, 10, 10, 10, 10])
    assert bad == 1
    assert kl.tolist() == [10, 14, 12, 10, 10]
