"""One speculative round on the GDN layers — verify, accept, rollback — on preallocated device
buffers. Plumbing only: every step is a call into libgdnspec (``_lib``); torch supplies the device
memory and the stream.
"""
import torch

from . import _lib
from .inputs import Workload


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
                                   W=w.W, io_dtype=w.io_dtype)
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

    def launches_per_step(self):
        """Kernel launches one step() enqueues (verify 1, accept 2 or 3, rollback 1)."""
        return 1 + (3 if self.mode == _lib.SPEC_MODE_SAMPLE and self.w.accept != "tree" else 2) + 1

    def check_status(self):
        torch.cuda.synchronize(self.device)
        v = int(self.status.item())
        if v:
            raise _lib.GdnError("device status 0x%x: %s" % (v, _lib.decode_status(v)))
