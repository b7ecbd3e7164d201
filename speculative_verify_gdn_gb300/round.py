"""One speculative round on the GDN layers — verify, accept, rollback — on preallocated device
buffers. Plumbing only: every step is a call into libgdnspec (``_lib``); torch supplies the device
memory and the stream.
"""
import torch

from . import _lib
from .inputs import Workload


def fused_in_one_kernel(w: Workload):
    """Whether gdn_rollback_verify runs as one kernel for this workload (else as two calls)."""
    import torch as _t
    return (w.io_dtype == _t.bfloat16 and w.D == 128 and w.N <= 8 and w.accept != "tree"
            and w.Hv in (w.Hk, 2 * w.Hk) and not w.gate_dk)


class SpecRound:
    """Owns the per-round outputs (o, tape, accept results, workspace, status) of a workload.

    The caller owns the model-side tensors (conv weights, recurrent state, conv state) and the
    round's inputs (qkv, g, beta, logits, drafts / tree).
    """

    def __init__(self, w: Workload, device="cuda"):
        self.w = w
        dev = torch.device(device)
        self.device = dev
        self.shape = _lib.GdnShape(L=w.L, B=w.B, T=w.N, Hk=w.Hk, Hv=w.Hv, Dk=w.D, Dv=w.D,
                                   W=w.W, io_dtype=w.io_dtype, gate_dk=w.gate_dk)
        sh = self.shape
        self.out = torch.empty(sh.out_shape(), dtype=w.io_dtype, device=dev)
        self.tape_delta = torch.empty(sh.out_shape(), dtype=torch.float32, device=dev)
        self.tape_k = torch.empty(sh.tape_k_shape(), dtype=torch.float32, device=dev)
        self.n_acc = torch.zeros(w.B, dtype=torch.int32, device=dev)
        P = w.P
        self.out_tokens = torch.empty((w.B, P + 1), dtype=torch.int32, device=dev)
        self.path = torch.empty((w.B, P), dtype=torch.int32, device=dev) if w.accept == "tree" \
            else None
        self.mode = _lib.SPEC_MODE_SAMPLE if w.accept == "sample" else _lib.SPEC_MODE_GREEDY
        ldt = torch.float32 if w.io_dtype == torch.float32 else torch.bfloat16
        nbytes = _lib.workspace_bytes(w.B, w.N, w.V, self.mode, ldt)
        self.workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    # ---------------------------------------------------------------- the three calls
    def verify(self, qkv, conv_w, conv_state, g, beta, state, parent=None, stream=None):
        _lib.verify(self.shape, qkv, conv_w, conv_state, g, beta, state, self.out,
                    self.tape_delta, self.tape_k, status=self.status, parent=parent,
                    stream=stream)

    def accept(self, logits, drafts, round_=0, seed=0, parent=None, stream=None):
        w = self.w
        if w.accept == "tree":
            _lib.spec_accept_tree(logits, parent, drafts, self.path, self.n_acc,
                                  self.out_tokens, self.workspace, status=self.status,
                                  stream=stream)
        else:
            _lib.spec_accept(logits, drafts, self.n_acc, self.out_tokens, self.workspace,
                             mode=self.mode, temperature=w.temperature, seed=seed,
                             round_=round_, status=self.status, stream=stream)

    def rollback(self, qkv, g, state, conv_state, stream=None):
        _lib.rollback(self.shape, self.n_acc, self.tape_delta, self.tape_k, g, qkv, state,
                      conv_state, status=self.status, path=self.path, stream=stream)

    def step(self, qkv, g, beta, logits, drafts, conv_w, state, conv_state, round_=0, seed=0,
             parent=None, stream=None):
        """verify -> accept -> rollback; state and conv_state are updated in place."""
        self.verify(qkv, conv_w, conv_state, g, beta, state, parent=parent, stream=stream)
        self.accept(logits, drafts, round_=round_, seed=seed, parent=parent, stream=stream)
        self.rollback(qkv, g, state, conv_state, stream=stream)

    # ---------------------------------------------------------------- fused round loop
    def rollback_verify(self, qkv, conv_w, conv_state, g, beta, state, stream=None):
        """gdn_rollback_verify: commit the previous fused round (its accept result, tape, qkv, g)
        and verify this one. The caller keeps qkv and g alive and unchanged until the next call
        (they are the next commit's tape)."""
        if self.w.accept == "tree":
            raise ValueError("the fused round loop serves chains; trees use step()")
        if not hasattr(self, "_prev"):
            self._alloc_fused()
        prev, cur = self._prev, self._cur
        first = prev["qkv"] is None          # nothing to commit: n_acc_prev is zero
        _lib.rollback_verify(self.shape, prev["n_acc"], prev["tape_delta"], prev["tape_k"],
                             g if first else prev["g"], qkv if first else prev["qkv"], qkv,
                             conv_w, conv_state, g, beta, state, self.out, cur["tape_delta"],
                             cur["tape_k"], status=self.status, stream=stream)
        self.tape_delta, self.tape_k, self.n_acc = cur["tape_delta"], cur["tape_k"], cur["n_acc"]
        cur["g"], cur["qkv"] = g, qkv
        self._prev, self._cur = cur, prev

    def step_fused(self, qkv, g, beta, logits, drafts, conv_w, state, conv_state, round_=0,
                   seed=0, stream=None):
        """rollback_verify -> accept. The state lags one round behind: flush() after the last."""
        self.rollback_verify(qkv, conv_w, conv_state, g, beta, state, stream=stream)
        self.accept(logits, drafts, round_=round_, seed=seed, stream=stream)

    def flush(self, state, conv_state, stream=None):
        """Commit the last step_fused round (gdn_rollback with its accept result)."""
        if not hasattr(self, "_prev") or self._prev["qkv"] is None:
            return
        p = self._prev
        _lib.rollback(self.shape, p["n_acc"], p["tape_delta"], p["tape_k"], p["g"], p["qkv"],
                      state, conv_state, status=self.status, stream=stream)
        p["n_acc"].zero_()
        p["qkv"] = p["g"] = None

    def _alloc_fused(self):
        sh, dev = self.shape, self.device
        def buf():
            return {"tape_delta": torch.empty(sh.out_shape(), dtype=torch.float32, device=dev),
                    "tape_k": torch.empty(sh.tape_k_shape(), dtype=torch.float32, device=dev),
                    "n_acc": torch.zeros(self.w.B, dtype=torch.int32, device=dev),
                    "g": None, "qkv": None}
        self._prev, self._cur = buf(), buf()

    def launches_per_step(self, fused=False):
        """Kernel launches one step() (verify 1, accept 1 to 3, rollback 1) or one step_fused()
        (rollback_verify 1, accept 1 to 3) enqueues, for shapes the fused kernel serves: sampling
        accept is one cluster kernel from a vocabulary of 8192 on (three kernels below), greedy and
        tree accept two."""
        if self.mode == _lib.SPEC_MODE_SAMPLE and self.w.accept != "tree":
            acc = 1 if self.w.V >= 8192 else 3
        else:
            acc = 2
        return (1 if fused and fused_in_one_kernel(self.w) else 2) + acc

    def check_status(self):
        torch.cuda.synchronize(self.device)
        _lib.status_check(int(self.status.item()))
