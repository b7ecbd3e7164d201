"""ctypes binding of the C oracle (oracle.c). Test infrastructure only.

Every array argument is converted to a C-contiguous numpy array of the dtype the C side reads
(float64 tensors, float32 logits, int32 indices); results come back as new numpy arrays.
"""
import ctypes as ct
from dataclasses import dataclass

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        _lib = ct.CDLL(_build.build())
        P = ct.c_void_p
        i32, i64, u32, u64, f32 = ct.c_int32, ct.c_int64, ct.c_uint32, ct.c_uint64, ct.c_float
        _lib.oracle_verify.argtypes = [P] * 12
        _lib.oracle_verify.restype = None
        _lib.oracle_rollback.argtypes = [P, P, ct.c_int] + [P] * 7
        _lib.oracle_rollback.restype = ct.c_int
        _lib.oracle_argmax.argtypes = [P, ct.c_int]
        _lib.oracle_argmax.restype = ct.c_int
        _lib.oracle_accept_greedy.argtypes = [ct.c_int] * 3 + [i64, i64, P, P, P, P]
        _lib.oracle_accept_greedy.restype = ct.c_int
        _lib.oracle_exp2_spec.argtypes = [f32]
        _lib.oracle_exp2_spec.restype = f32
        _lib.oracle_scale_c.argtypes = [f32]
        _lib.oracle_scale_c.restype = f32
        _lib.oracle_weights.argtypes = [P, ct.c_int, f32, ct.c_int, P]
        _lib.oracle_weights.restype = u64
        _lib.oracle_philox4x32_10.argtypes = [P, P, P]
        _lib.oracle_philox4x32_10.restype = None
        _lib.oracle_draw.argtypes = [u64, u32, u32, u32, u32, u64]
        _lib.oracle_draw.restype = u64
        _lib.oracle_accept_sample.argtypes = ([ct.c_int] * 3 + [i64, i64, P, P, f32, u64, u64,
                                                                 P, P])
        _lib.oracle_accept_sample.restype = ct.c_int
        _lib.oracle_accept_tree.argtypes = ([ct.c_int] * 3 + [i64, i64, P, P, P, ct.c_int,
                                                               P, P, P])
        _lib.oracle_accept_tree.restype = ct.c_int
        _lib.oracle_attn_verify.argtypes = [P] * 8
        _lib.oracle_attn_verify.restype = ct.c_int
        _lib.oracle_attn_truncate.argtypes = [ct.c_int, ct.c_int, P, P]
        _lib.oracle_attn_truncate.restype = ct.c_int
        _lib.oracle_set_threads.argtypes = [ct.c_int]
        _lib.oracle_set_threads.restype = None
        _lib.oracle_get_threads.argtypes = []
        _lib.oracle_get_threads.restype = ct.c_int
        _lib.oracle_openmp.argtypes = []
        _lib.oracle_openmp.restype = ct.c_int
        del i32
    return _lib


def set_threads(n):
    """Threads for the loops over independent units (results do not depend on it). Returns the
    count in effect: 1 when the library was built without OpenMP."""
    lib = _load()
    lib.oracle_set_threads(int(n))
    return lib.oracle_get_threads() if lib.oracle_openmp() else 1


class _CDims(ct.Structure):
    _fields_ = [(n, ct.c_int) for n in ("L", "B", "T", "Hk", "Hv", "Dk", "Dv", "W", "C",
                                         "act_silu", "gate_dk")] + [("qk_scale", ct.c_double),
                                                                    ("l2_eps", ct.c_double)]


@dataclass
class OracleDims:
    L: int
    B: int
    T: int
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    W: int
    act_silu: bool = True
    qk_scale: float = 1.0
    l2_eps: float = 1e-6

    @property
    def C(self):
        return 2 * self.Hk * self.Dk + self.Hv * self.Dv

    def c(self, gate_dk=False):
        return _CDims(self.L, self.B, self.T, self.Hk, self.Hv, self.Dk, self.Dv, self.W, self.C,
                      1 if self.act_silu else 0, 1 if gate_dk else 0, float(self.qk_scale),
                      float(self.l2_eps))


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a):
    return None if a is None else a.ctypes.data_as(ct.c_void_p)


def verify(dims: OracleDims, qkv, conv_w, conv_state, g, beta, state, parent=None,
           node_states=False):
    """Returns dict(out, tape_delta, tape_k[, node_state]) as float64 arrays.

    Shapes as the C ABI: qkv [L,B,T,C], conv_w [L,C,W], conv_state [L,B,W-1,C], g/beta
    [L,B,T,Hv], state [L,B,Hv,Dv,Dk] (row-major S); parent [B,T] int32 or None for the chain.
    """
    lib = _load()
    d = dims
    qkv, conv_w, conv_state = _f64(qkv), _f64(conv_w), _f64(conv_state)
    g, beta, state = _f64(g), _f64(beta), _f64(state)
    assert qkv.shape == (d.L, d.B, d.T, d.C), qkv.shape
    assert conv_w.shape == (d.L, d.C, d.W)
    assert conv_state.shape == (d.L, d.B, d.W - 1, d.C)
    # g per value head [L,B,T,Hv], or per key channel [L,B,T,Hv,Dk]
    gate_dk = g.ndim == 5
    assert g.shape == ((d.L, d.B, d.T, d.Hv, d.Dk) if gate_dk else (d.L, d.B, d.T, d.Hv)), g.shape
    assert beta.shape == (d.L, d.B, d.T, d.Hv)
    assert state.shape == (d.L, d.B, d.Hv, d.Dv, d.Dk)
    par = None if parent is None else _i32(parent)
    if par is not None:
        assert par.shape == (d.B, d.T)
    out = np.zeros((d.L, d.B, d.T, d.Hv, d.Dv))
    tdl = np.zeros_like(out)
    tk = np.zeros((d.L, d.B, d.T, d.Hk, d.Dk))
    ns = np.zeros((d.L, d.B, d.T, d.Hv, d.Dv, d.Dk)) if node_states else None
    cd = d.c(gate_dk)
    lib.oracle_verify(ct.byref(cd), _p(par), _p(qkv), _p(conv_w), _p(conv_state), _p(g),
                      _p(beta), _p(state), _p(out), _p(tdl), _p(tk), _p(ns))
    res = dict(out=out, tape_delta=tdl, tape_k=tk)
    if node_states:
        res["node_state"] = ns
    return res


def rollback(dims: OracleDims, n_acc, tape_delta, tape_k, g, qkv, state, conv_state, path=None):
    """Tape replay. Returns (state, conv_state, bad_bits) with new arrays (inputs untouched)."""
    lib = _load()
    d = dims
    n_acc = _i32(n_acc)
    st = _f64(state).copy()
    cs = _f64(conv_state).copy()
    pth = None if path is None else _i32(path)
    P = 0 if pth is None else pth.shape[1]
    g = _f64(g)
    cd = d.c(g.ndim == 5)
    bad = lib.oracle_rollback(ct.byref(cd), _p(pth), P, _p(n_acc), _p(_f64(tape_delta)),
                              _p(_f64(tape_k)), _p(g), _p(_f64(qkv)), _p(st), _p(cs))
    return st, cs, bad


def argmax(row):
    row = _f32(row)
    return _load().oracle_argmax(_p(row), row.shape[-1])


def _logit_view(logits):
    lg = _f32(logits)
    B, R, V = lg.shape
    return lg, B, R, V


def accept_greedy(logits, drafts):
    """logits [B, N+1, V] (float32 values), drafts [B, N] -> (n_acc [B], out [B, N+1], bad)."""
    lg, B, R, V = _logit_view(logits)
    N = R - 1
    dr = _i32(drafts).reshape(B, N)
    n = np.zeros(B, np.int32)
    out = np.zeros((B, N + 1), np.int32)
    bad = _load().oracle_accept_greedy(B, N, V, V, R * V, _p(lg), _p(dr), _p(n), _p(out))
    return n, out, bad


def accept_sample(logits, drafts, temperature, seed, round_, seq_shared=False, B=None):
    """Leviathan sampling. logits [B, N+1, V] (or [1, N+1, V] with seq_shared=True and B given,
    every sequence reading the same rows). Returns (n_acc, out, bad)."""
    lg, Bl, R, V = _logit_view(logits)
    N = R - 1
    if seq_shared:
        assert Bl == 1 and B is not None
        seq_stride = 0
    else:
        B = Bl
        seq_stride = R * V
    dr = _i32(drafts).reshape(B, N)
    n = np.zeros(B, np.int32)
    out = np.zeros((B, N + 1), np.int32)
    bad = _load().oracle_accept_sample(B, N, V, V, seq_stride, _p(lg), _p(dr),
                                       ct.c_float(np.float32(temperature)), int(seed),
                                       int(round_), _p(n), _p(out))
    return n, out, bad


def accept_tree(logits, parent, tokens, P):
    """logits [B, T+1, V]; parent, tokens [B, T] -> (path [B,P], n_acc [B], out [B,P+1], bad)."""
    lg, B, R, V = _logit_view(logits)
    T = R - 1
    par = _i32(parent).reshape(B, T)
    tok = _i32(tokens).reshape(B, T)
    path = np.zeros((B, P), np.int32)
    n = np.zeros(B, np.int32)
    out = np.zeros((B, P + 1), np.int32)
    bad = _load().oracle_accept_tree(B, T, V, V, R * V, _p(lg), _p(par), _p(tok), int(P),
                                     _p(path), _p(n), _p(out))
    return path, n, out, bad


def exp2_spec(x):
    lib = _load()
    x = np.asarray(x, np.float32)
    flat = np.array([lib.oracle_exp2_spec(ct.c_float(v)) for v in x.ravel()], np.float32)
    return flat.reshape(x.shape)


def scale_c(temperature):
    return np.float32(_load().oracle_scale_c(ct.c_float(np.float32(temperature))))


def weights(row, temperature, ban=-1):
    """Integer weights of one row and their sum Z."""
    lib = _load()
    row = _f32(row)
    w = np.zeros(row.shape[-1], np.uint64)
    Z = lib.oracle_weights(_p(row), row.shape[-1], ct.c_float(scale_c(temperature)), int(ban),
                           _p(w))
    return w, int(Z)


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(np.asarray(ctr, np.uint32))
    k = np.ascontiguousarray(np.asarray(key, np.uint32))
    o = np.zeros(4, np.uint32)
    _load().oracle_philox4x32_10(_p(c), _p(k), _p(o))
    return o


def draw(seed, round_, seq, row, purpose, Z):
    return int(_load().oracle_draw(int(seed), int(round_) & 0xFFFFFFFF, int(seq), int(row),
                                   int(purpose), int(Z)))


def accept_stats(calls, N):
    """Acceptance counters over a sequence of accept calls (colibrì ch.08 §4.1 counts proposals
    and acceptances): proposed = Σ B·N, accepted = Σ n, hist[k] = #sequences with n = k. A count
    outside [0, N] adds only its N proposals; the returned flag says whether any was seen."""
    proposed, accepted, hist, bad = 0, 0, [0] * (N + 1), False
    for n_acc in calls:
        for n in [int(x) for x in n_acc]:
            proposed += N
            if n < 0 or n > N:
                bad = True
                continue
            accepted += n
            hist[n] += 1
    return proposed, accepted, hist, bad


def adaptive_enabled(proposed, accepted, min_proposed=24, num=1, den=10):
    """The off-switch rule as the page states it: drafting stops once at least min_proposed
    drafts were proposed and accepted * 10 < proposed (num / den generalises the 1/10)."""
    if proposed < min_proposed:
        return True
    return not (accepted * den < proposed * num)


class _CAttnDims(ct.Structure):
    _fields_ = [(n, ct.c_int) for n in ("L", "B", "T", "Hq", "Hkv", "D", "ctx")] + [
        ("scale", ct.c_double)]


@dataclass
class AttnDims:
    """Attention-layer shapes: L layers, B sequences, T verify positions, Hq query heads over Hkv
    kv heads (query head h reads kv head h // (Hq / Hkv)), head dim D, cache capacity ctx rows;
    scale defaults to 1 / sqrt(D)."""
    L: int
    B: int
    T: int
    Hq: int
    Hkv: int
    D: int
    ctx: int
    scale: float = None

    def c(self):
        sc = self.scale if self.scale is not None else 1.0 / np.sqrt(self.D)
        return _CAttnDims(self.L, self.B, self.T, self.Hq, self.Hkv, self.D, self.ctx, float(sc))


def attn_verify(dims: AttnDims, kv_len, q, k_new, v_new, k_cache, v_cache):
    """Full-attention verify. q [L,B,T,Hq,D], k_new / v_new [L,B,T,Hkv,D], caches
    [L,B,Hkv,ctx,D] token-major, kv_len [B]. Returns (out [L,B,T,Hq,D], k_cache, v_cache (new
    arrays with the T rows appended), bad)."""
    d = dims
    q, k_new, v_new = _f64(q), _f64(k_new), _f64(v_new)
    kc, vc = _f64(k_cache).copy(), _f64(v_cache).copy()
    assert q.shape == (d.L, d.B, d.T, d.Hq, d.D), q.shape
    assert k_new.shape == v_new.shape == (d.L, d.B, d.T, d.Hkv, d.D)
    assert kc.shape == vc.shape == (d.L, d.B, d.Hkv, d.ctx, d.D)
    assert d.Hq % d.Hkv == 0
    n = _i32(kv_len)
    out = np.zeros_like(q)
    cd = d.c()
    bad = _load().oracle_attn_verify(ct.byref(cd), _p(n), _p(q), _p(k_new), _p(v_new), _p(kc),
                                     _p(vc), _p(out))
    return out, kc, vc, bad


def attn_truncate(T, n_acc, kv_len):
    """KV truncation: returns (kv_len + n_acc where 0 <= n <= T, bad)."""
    n = _i32(n_acc)
    kl = _i32(kv_len).copy()
    bad = _load().oracle_attn_truncate(len(kl), int(T), _p(n), _p(kl))
    return kl, bad

