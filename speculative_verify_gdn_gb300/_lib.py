"""ctypes binding of libgdnspec (include/gdnspec.h). Argument marshalling only: every step of the
path runs in the library's CUDA kernels. The library must be built (``build.py``); a missing
library raises at first use — there is no fallback.

All tensors are torch CUDA tensors, contiguous, with the dtypes and layouts of the C header;
calls are enqueued on ``torch.cuda.current_stream()`` unless a stream is given.
"""
import ctypes as ct
import os
from dataclasses import dataclass

import torch

from . import build as _build

GDN_OK = 0
GDN_ERR_DEVICE_STATUS = 4
GDN_DTYPE_F32 = 0
GDN_DTYPE_BF16 = 1
SPEC_MODE_GREEDY = 0
SPEC_MODE_SAMPLE = 1

STATUS_BITS = {
    0x1: "BAD_NACC",
    0x2: "BAD_PARENT",
    0x4: "BAD_TOKEN",
    0x8: "BAD_PATH",
    0x10: "EMPTY_DIST",
    0x20: "WAIT_TIMEOUT",
    0x40: "BAD_LEN",
}

# exported entry points of include/gdnspec.h
EXPORTS = ("gdn_verify", "gdn_verify_tree", "gdn_rollback", "gdn_rollback_path",
           "gdn_rollback_verify", "gdn_tape_bytes", "spec_accept", "spec_workspace_bytes", "spec_accept_tree",
           "spec_accept_static", "spec_stats_accumulate", "attn_verify", "attn_workspace_bytes",
           "attn_truncate", "gdn_last_error", "gdn_status_check", "gdn_set_wait_limit_ns")


class GdnError(RuntimeError):
    pass


class _Dims(ct.Structure):
    _fields_ = [(n, ct.c_int32) for n in ("L", "B", "T", "Hk", "Hv", "Dk", "Dv", "W", "C",
                                           "io_dtype")] + [("qk_scale", ct.c_float),
                                                           ("l2_eps", ct.c_float),
                                                           ("gate_dk", ct.c_int32)]


class _AttnDims(ct.Structure):
    _fields_ = [(n, ct.c_int32) for n in ("L", "B", "T", "Hq", "Hkv", "D", "ctx")] + [
        ("scale", ct.c_float)]


class _SpecDims(ct.Structure):
    _fields_ = [("B", ct.c_int32), ("N", ct.c_int32), ("V", ct.c_int32), ("dtype", ct.c_int32),
                ("row_stride", ct.c_int64), ("seq_stride", ct.c_int64)]


_lib = None


def library_path():
    return _build.LIB


def load(require_file=True):
    """Load libgdnspec.so (built in-tree). Raises if it does not exist."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise GdnError("libgdnspec.so is not built (%s): run "
                       "python -m speculative_verify_gdn_gb300.build" % path)
    lib = ct.CDLL(path)
    P, i32, u64, f32, sz = ct.c_void_p, ct.c_int32, ct.c_uint64, ct.c_float, ct.c_size_t
    lib.gdn_verify.argtypes = [P] * 12
    lib.gdn_verify_tree.argtypes = [P] * 13
    lib.gdn_rollback.argtypes = [P] * 10
    lib.gdn_rollback_path.argtypes = [P, P, i32] + [P] * 9
    lib.gdn_rollback_verify.argtypes = [P] * 17
    for f in (lib.gdn_verify, lib.gdn_verify_tree, lib.gdn_rollback, lib.gdn_rollback_path,
              lib.gdn_rollback_verify):
        f.restype = ct.c_int
    lib.gdn_tape_bytes.argtypes = [P]
    lib.gdn_tape_bytes.restype = sz
    lib.spec_accept.argtypes = [P, P, P, i32, f32, u64, u64, P, sz, P, P, P, P]
    lib.spec_accept.restype = ct.c_int
    lib.spec_workspace_bytes.argtypes = [P, i32]
    lib.spec_workspace_bytes.restype = sz
    lib.spec_accept_tree.argtypes = [P, P, P, P, i32, P, sz, P, P, P, P, P]
    lib.spec_accept_tree.restype = ct.c_int
    lib.spec_accept_static.argtypes = [P, P, P, i32, f32, u64, u64, P, P, P, P]
    lib.spec_accept_static.restype = ct.c_int
    lib.spec_stats_accumulate.argtypes = [i32, i32, P, P, P, P]
    lib.spec_stats_accumulate.restype = ct.c_int
    lib.attn_verify.argtypes = [P] * 9 + [sz, P, P]
    lib.attn_verify.restype = ct.c_int
    lib.attn_workspace_bytes.argtypes = [P]
    lib.attn_workspace_bytes.restype = sz
    lib.attn_truncate.argtypes = [i32, i32, P, P, P, P]
    lib.attn_truncate.restype = ct.c_int
    lib.gdn_last_error.argtypes = []
    lib.gdn_last_error.restype = ct.c_char_p
    lib.gdn_status_check.argtypes = [ct.c_uint32]
    lib.gdn_status_check.restype = ct.c_int
    lib.gdn_set_wait_limit_ns.argtypes = [ct.c_uint64]
    lib.gdn_set_wait_limit_ns.restype = ct.c_int
    _lib = lib
    return lib


def last_error():
    return load().gdn_last_error().decode()


def _check(rc, what):
    if rc != GDN_OK:
        raise GdnError("%s failed (code %d): %s" % (what, rc, last_error()))


@dataclass
class GdnShape:
    """Shapes of one gdn_verify / gdn_rollback call (see gdn_dims in include/gdnspec.h)."""
    L: int
    B: int
    T: int
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    W: int = 4
    io_dtype: torch.dtype = torch.bfloat16
    qk_scale: float = 1.0
    l2_eps: float = 1e-6
    gate_dk: bool = False      # g per key channel [L, B, T, Hv, Dk]

    @property
    def C(self):
        return 2 * self.Hk * self.Dk + self.Hv * self.Dv

    def c(self):
        dt = GDN_DTYPE_BF16 if self.io_dtype == torch.bfloat16 else GDN_DTYPE_F32
        return _Dims(self.L, self.B, self.T, self.Hk, self.Hv, self.Dk, self.Dv, self.W, self.C,
                     dt, self.qk_scale, self.l2_eps, 1 if self.gate_dk else 0)

    # expected tensor shapes
    def qkv_shape(self):
        return (self.L, self.B, self.T, self.C)

    def conv_w_shape(self):
        return (self.L, self.C, self.W)

    def conv_state_shape(self):
        return (self.L, self.B, self.W - 1, self.C)

    def gate_shape(self):
        """Shape of g: per value head, or per key channel when gate_dk."""
        return (self.L, self.B, self.T, self.Hv) + ((self.Dk,) if self.gate_dk else ())

    def beta_shape(self):
        return (self.L, self.B, self.T, self.Hv)

    def state_shape(self):
        return (self.L, self.B, self.Hv, self.Dv, self.Dk)

    def out_shape(self):
        return (self.L, self.B, self.T, self.Hv, self.Dv)

    def tape_k_shape(self):
        return (self.L, self.B, self.T, self.Hk, self.Dk)


def _ptr(t, dtype=None, shape=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise GdnError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise GdnError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise GdnError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise GdnError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return ct.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ct.c_void_p(s.cuda_stream)


def tape_bytes(shape: GdnShape):
    return int(load().gdn_tape_bytes(ct.byref(shape.c())))


def verify(shape: GdnShape, qkv, conv_w, conv_state, g, beta, state, out, tape_delta, tape_k,
           status=None, parent=None, stream=None):
    """gdn_verify (parent None) or gdn_verify_tree."""
    lib = load()
    io = shape.io_dtype
    f32 = torch.float32
    d = shape.c()
    args = [_ptr(qkv, io, shape.qkv_shape(), "qkv"),
            _ptr(conv_w, io, shape.conv_w_shape(), "conv_w"),
            _ptr(conv_state, io, shape.conv_state_shape(), "conv_state"),
            _ptr(g, f32, shape.gate_shape(), "g"), _ptr(beta, f32, shape.beta_shape(), "beta"),
            _ptr(state, f32, shape.state_shape(), "state"),
            _ptr(out, io, shape.out_shape(), "out"),
            _ptr(tape_delta, f32, shape.out_shape(), "tape_delta"),
            _ptr(tape_k, f32, shape.tape_k_shape(), "tape_k"),
            _ptr(status, torch.int32, None, "status"), _stream(stream)]
    if parent is None:
        _check(lib.gdn_verify(ct.byref(d), *args), "gdn_verify")
    else:
        par = _ptr(parent, torch.int32, (shape.B, shape.T), "parent")
        _check(lib.gdn_verify_tree(ct.byref(d), par, *args), "gdn_verify_tree")


def rollback(shape: GdnShape, n_acc, tape_delta, tape_k, g, qkv, state, conv_state, status=None,
             path=None, stream=None):
    """gdn_rollback (path None) or gdn_rollback_path (path [B, P] int32)."""
    lib = load()
    io = shape.io_dtype
    f32 = torch.float32
    d = shape.c()
    args = [_ptr(n_acc, torch.int32, (shape.B,), "n_acc"),
            _ptr(tape_delta, f32, shape.out_shape(), "tape_delta"),
            _ptr(tape_k, f32, shape.tape_k_shape(), "tape_k"),
            _ptr(g, f32, shape.gate_shape(), "g"), _ptr(qkv, io, shape.qkv_shape(), "qkv"),
            _ptr(state, f32, shape.state_shape(), "state"),
            _ptr(conv_state, io, shape.conv_state_shape(), "conv_state"),
            _ptr(status, torch.int32, None, "status"), _stream(stream)]
    if path is None:
        _check(lib.gdn_rollback(ct.byref(d), *args), "gdn_rollback")
    else:
        if path.dim() != 2 or path.shape[0] != shape.B:
            raise GdnError("path must be [B, P]")
        pp = _ptr(path, torch.int32, None, "path")
        _check(lib.gdn_rollback_path(ct.byref(d), pp, int(path.shape[1]), *args),
               "gdn_rollback_path")


def rollback_verify(shape: GdnShape, n_acc_prev, tape_delta_prev, tape_k_prev, g_prev, qkv_prev,
                    qkv, conv_w, conv_state, g, beta, state, out, tape_delta, tape_k,
                    status=None, stream=None):
    """gdn_rollback_verify: the previous round's rollback and this round's verify in one call."""
    lib = load()
    io = shape.io_dtype
    f32 = torch.float32
    d = shape.c()
    args = [_ptr(n_acc_prev, torch.int32, (shape.B,), "n_acc_prev"),
            _ptr(tape_delta_prev, f32, shape.out_shape(), "tape_delta_prev"),
            _ptr(tape_k_prev, f32, shape.tape_k_shape(), "tape_k_prev"),
            _ptr(g_prev, f32, shape.gate_shape(), "g_prev"),
            _ptr(qkv_prev, io, shape.qkv_shape(), "qkv_prev"),
            _ptr(qkv, io, shape.qkv_shape(), "qkv"),
            _ptr(conv_w, io, shape.conv_w_shape(), "conv_w"),
            _ptr(conv_state, io, shape.conv_state_shape(), "conv_state"),
            _ptr(g, f32, shape.gate_shape(), "g"), _ptr(beta, f32, shape.beta_shape(), "beta"),
            _ptr(state, f32, shape.state_shape(), "state"),
            _ptr(out, io, shape.out_shape(), "out"),
            _ptr(tape_delta, f32, shape.out_shape(), "tape_delta"),
            _ptr(tape_k, f32, shape.tape_k_shape(), "tape_k"),
            _ptr(status, torch.int32, None, "status"), _stream(stream)]
    _check(lib.gdn_rollback_verify(ct.byref(d), *args), "gdn_rollback_verify")


def _spec_dims(logits, B=None, V=None):
    """logits [B, R, Vpad] (or [1, R, Vpad] broadcast to B sequences with B given); the first V
    entries of each row are the vocabulary (V defaults to Vpad)."""
    if logits.dim() != 3:
        raise GdnError("logits must be [B, rows, V]")
    Bl, R, Vpad = logits.shape
    V = Vpad if V is None else int(V)
    if not 0 < V <= Vpad:
        raise GdnError("V must be in (0, row length]")
    dt = GDN_DTYPE_BF16 if logits.dtype == torch.bfloat16 else GDN_DTYPE_F32
    if logits.dtype not in (torch.bfloat16, torch.float32):
        raise GdnError("logits must be bf16 or fp32")
    if B is None:
        B, seq_stride = Bl, R * Vpad
    else:
        if Bl != 1:
            raise GdnError("broadcast logits must have a leading dim of 1")
        seq_stride = 0
    return _SpecDims(B, R - 1, V, dt, Vpad, seq_stride)


def workspace_bytes(B, N, V, mode=SPEC_MODE_GREEDY, dtype=torch.bfloat16):
    dt = GDN_DTYPE_BF16 if dtype == torch.bfloat16 else GDN_DTYPE_F32
    vec = 8 if dt == GDN_DTYPE_BF16 else 4
    d = _SpecDims(B, N, V, dt, (V + vec - 1) // vec * vec, 0)
    return int(load().spec_workspace_bytes(ct.byref(d), mode))


def spec_accept(logits, drafts, n_acc, out_tokens, workspace, mode=SPEC_MODE_GREEDY,
                temperature=0.0, seed=0, round_=0, status=None, stream=None, broadcast_B=None,
                V=None):
    lib = load()
    d = _spec_dims(logits, broadcast_B, V)
    B, N = d.B, d.N
    if workspace.dtype != torch.uint8:
        raise GdnError("workspace must be a uint8 tensor")
    rc = lib.spec_accept(ct.byref(d), _ptr(logits, None, None, "logits"),
                         _ptr(drafts, torch.int32, (B, N), "drafts"), int(mode),
                         ct.c_float(float(temperature)), int(seed) & (2**64 - 1),
                         int(round_) & (2**64 - 1), _ptr(workspace, None, None, "workspace"),
                         workspace.numel(), _ptr(n_acc, torch.int32, (B,), "n_acc"),
                         _ptr(out_tokens, torch.int32, (B, N + 1), "out_tokens"),
                         _ptr(status, torch.int32, None, "status"), _stream(stream))
    _check(rc, "spec_accept")


def spec_stats_accumulate(n_acc, N, stats, status=None, stream=None):
    """spec_stats_accumulate: stats (int64 [N + 3], holding the uint64 counters) += proposed,
    accepted and the histogram of accepted lengths of this call's n_acc ([B] int32)."""
    B = int(n_acc.shape[0]) if n_acc.dim() == 1 else -1
    rc = load().spec_stats_accumulate(B, int(N), _ptr(n_acc, torch.int32, (B,), "n_acc"),
                                      _ptr(stats, torch.int64, (int(N) + 3,), "stats"),
                                      _ptr(status, torch.int32, None, "status"), _stream(stream))
    _check(rc, "spec_stats_accumulate")


def spec_accept_tree(logits, parent, tokens, path, n_acc, out_tokens, workspace, status=None,
                     stream=None, V=None):
    lib = load()
    d = _spec_dims(logits, None, V)
    B, T = d.B, d.N
    P = int(path.shape[1])
    rc = lib.spec_accept_tree(ct.byref(d), _ptr(logits, None, None, "logits"),
                              _ptr(parent, torch.int32, (B, T), "parent"),
                              _ptr(tokens, torch.int32, (B, T), "tokens"), P,
                              _ptr(workspace, None, None, "workspace"), workspace.numel(),
                              _ptr(path, torch.int32, (B, P), "path"),
                              _ptr(n_acc, torch.int32, (B,), "n_acc"),
                              _ptr(out_tokens, torch.int32, (B, P + 1), "out_tokens"),
                              _ptr(status, torch.int32, None, "status"), _stream(stream))
    _check(rc, "spec_accept_tree")


def decode_status(value):
    value = int(value) & 0xFFFFFFFF
    return [name for bit, name in STATUS_BITS.items() if value & bit]


def set_wait_limit_ns(ns):
    """Give-up time of the pipelined verify kernel's pipeline waits (0: the default second)."""
    _check(load().gdn_set_wait_limit_ns(int(ns)), "gdn_set_wait_limit_ns")


def status_check(value):
    """Raises GdnError (the library's GDN_ERR_DEVICE_STATUS message) for a non-zero status word
    read back after synchronising; host only."""
    _check(load().gdn_status_check(int(value) & 0xFFFFFFFF), "device status")


# ------------------------------------------------------------------ attention layers
@dataclass
class AttnShape:
    """Shapes of one attn_verify call (see attn_dims in include/gdnspec.h); scale defaults to
    1/sqrt(D)."""
    L: int
    B: int
    T: int
    Hq: int
    Hkv: int
    D: int
    ctx: int
    scale: float = None

    def c(self):
        sc = self.scale if self.scale is not None else 1.0 / self.D ** 0.5
        return _AttnDims(self.L, self.B, self.T, self.Hq, self.Hkv, self.D, self.ctx, sc)

    def q_shape(self):
        return (self.L, self.B, self.T, self.Hq, self.D)

    def kv_new_shape(self):
        return (self.L, self.B, self.T, self.Hkv, self.D)

    def k_cache_shape(self):
        return (self.L, self.B, self.Hkv, self.ctx, self.D)

    def vt_cache_shape(self):
        return (self.L, self.B, self.Hkv, self.ctx // 128, self.D, 128)


def vt_from_v(v_cache):
    """A token-major value cache [..., ctx, D] in the library's tile-transposed layout
    [..., ctx/128, D, 128] (layout plumbing: a view, a transpose and a copy)."""
    *lead, ctx, D = v_cache.shape
    return v_cache.reshape(*lead, ctx // 128, 128, D).transpose(-1, -2).contiguous()


def v_from_vt(vt_cache):
    """The inverse of vt_from_v: [..., ctx/128, D, 128] -> [..., ctx, D]."""
    *lead, nt, D, _ = vt_cache.shape
    return vt_cache.transpose(-1, -2).reshape(*lead, nt * 128, D)


def attn_workspace_bytes(shape: AttnShape):
    return int(load().attn_workspace_bytes(ct.byref(shape.c())))


def attn_verify(shape: AttnShape, q, k_new, v_new, k_cache, vt_cache, kv_len, out,
                workspace=None, status=None, stream=None):
    """attn_verify: append the T positions' k / v rows at kv_len and attend causally over the
    cache (kv_len itself is left for attn_truncate)."""
    lib = load()
    bf = torch.bfloat16
    d = shape.c()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = [_ptr(q, bf, shape.q_shape(), "q"),
            _ptr(k_new, bf, shape.kv_new_shape(), "k_new"),
            _ptr(v_new, bf, shape.kv_new_shape(), "v_new"),
            _ptr(k_cache, bf, shape.k_cache_shape(), "k_cache"),
            _ptr(vt_cache, bf, shape.vt_cache_shape(), "vt_cache"),
            _ptr(kv_len, torch.int32, (shape.B,), "kv_len"),
            _ptr(out, bf, shape.q_shape(), "out"),
            _ptr(workspace, None, None, "workspace"), ct.c_size_t(ws_bytes),
            _ptr(status, torch.int32, None, "status"), _stream(stream)]
    _check(lib.attn_verify(ct.byref(d), *args), "attn_verify")


def attn_truncate(n_acc, kv_len, T, status=None, stream=None):
    """attn_truncate: kv_len[b] += n_acc[b] on the device."""
    B = kv_len.shape[0]
    _check(load().attn_truncate(B, int(T), _ptr(n_acc, torch.int32, (B,), "n_acc"),
                                _ptr(kv_len, torch.int32, (B,), "kv_len"),
                                _ptr(status, torch.int32, None, "status"), _stream(stream)),
           "attn_truncate")

