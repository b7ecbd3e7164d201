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
