"""The give-up path of a bounded on-chip wait, made to run out on purpose.

Every mbarrier wait in the kernels spins for a limited wall time; one that runs out sets
GDN_STATUS_WAIT_TIMEOUT and the CTA runs to its end without waiting, so a stuck pipeline ends
with an error status instead of a hang. gdn_set_wait_limit_ns shortens the pipelined verify
kernel's pipeline waits (the waits that drain copies and tensor-core work before a CTA exits keep
their full second): at one nanosecond some wait always runs out. The status must say so, the
snapshot must be untouched (verify never writes it), and the next call at the default limit, in
the same process and context, must match the oracle again."""
import pytest
import torch

from speculative_verify_gdn_gb300 import _lib, inputs as I
from speculative_verify_gdn_gb300.round import SpecRound
from parity_util import to_dev
from test_gpu_parity import make_model, run_verify_case

pytestmark = pytest.mark.gpu


def test_pipeline_wait_gives_up_then_the_next_call_is_exact(gdnlib):
    # the smallest shape the pipelined kernel serves: bf16, d = 128, two value heads per key head
    w = I.custom(I.WORKLOADS[1], name="wait_timeout", L=1, B=1, N=4, Hk=2, Hv=4, D=128, V=64)
    cw, st, cs = make_model(w)
    qkv, g, beta = I.round_stream(w, 0, 0)
    dq, dcw, dcs, dg, db, dst = to_dev(qkv, cw, cs, g, beta, st)
    r = SpecRound(w)
    _lib.set_wait_limit_ns(1)
    try:
        r.verify(dq, dcw, dcs, dg, db, dst)
        torch.cuda.synchronize()
    finally:
        _lib.set_wait_limit_ns(0)
    v = int(r.status.item())
    assert v & 0x20, "no wait gave up (status %#x)" % v
    with pytest.raises(_lib.GdnError, match="WAIT_TIMEOUT"):
        _lib.status_check(v)
    assert torch.equal(dst.cpu(), st) and torch.equal(dcs.cpu(), cs)
    # the context is still usable and the default limit is back: parity with the oracle
    run_verify_case(w)
