"""Helpers shared by the GPU parity tests: run the oracle on the same seeded inputs and compare.

Tolerance for floating-point outputs (outputs o, the tape, states): elementwise
    |gpu - ref| <= 2e-3 * |ref| + 1e-5 * max|ref|          (values stored in fp32)
    |gpu - ref| <= 2e-3 * |ref| + 1e-5 * max|ref| + ulp_bf16(ref) / 2   (values stored in bf16)
with ref the oracle's unrounded fp64 value: 2e-3 relative is the computational error allowed, and
a bf16-stored value additionally carries the rounding to its I/O type (bf16 keeps 8 significant
bits, so that rounding alone reaches 2^-8 relative). Token ids and accepted counts are compared
bit-exactly.
"""
import numpy as np
import torch

import oracle
from oracle import OracleDims

RTOL = 2e-3
ATOL_FRAC = 1e-5


def f64(t):
    return t.detach().to("cpu").double().numpy()


def half_ulp_bf16(x):
    """Half the spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


def assert_close(gpu, ref, name, rtol=RTOL, atol_frac=ATOL_FRAC, bf16=False):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    if ref.size == 0:
        return
    scale = np.abs(ref).max()
    err = np.abs(gpu - ref)
    bound = rtol * np.abs(ref) + atol_frac * scale
    if bf16:
        bound = bound + half_ulp_bf16(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), ref.shape)
        raise AssertionError("%s: %d/%d elements out of tolerance; worst at %s: gpu=%r ref=%r "
                             "(max|ref|=%g)" % (name, bad.sum(), bad.size, i, gpu[i], ref[i],
                                                scale))


def oracle_dims(w, T=None, L=None, B=None):
    # the oracle reads the gate layout (per value head or per key channel) from g's rank
    return OracleDims(L=w.L if L is None else L, B=w.B if B is None else B,
                      T=w.N if T is None else T, Hk=w.Hk, Hv=w.Hv, Dk=w.D, Dv=w.D, W=w.W)


def oracle_verify(w, qkv, conv_w, conv_state, g, beta, state, parent=None, L=None, B=None):
    d = oracle_dims(w, L=L, B=B)
    return oracle.verify(d, f64(qkv), f64(conv_w), f64(conv_state), f64(g), f64(beta),
                         f64(state), parent=None if parent is None else parent.cpu().numpy())


def oracle_rollback(w, n_acc, ref, g, qkv, state, conv_state, path=None, L=None, B=None):
    d = oracle_dims(w, L=L, B=B)
    return oracle.rollback(d, np.asarray(n_acc, np.int32), ref["tape_delta"], ref["tape_k"],
                           f64(g), f64(qkv), f64(state), f64(conv_state),
                           path=None if path is None else np.asarray(path, np.int32))


def logits_f32(lg):
    return lg.detach().to("cpu").float().numpy()


def to_dev(*ts, device="cuda"):
    return [t.to(device).contiguous() for t in ts]


def state_copy(t):
    return t.clone()


__all__ = ["assert_close", "oracle_verify", "oracle_rollback", "oracle_dims", "f64",
           "logits_f32", "to_dev", "torch"]
