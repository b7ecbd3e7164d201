"""spec_accept_static: the accept entry point that allocates nothing (its scratch is a fixed array
in the library's device image). Some callers cannot allocate device memory — they only receive
device pointers from a host framework, or run where cudaMalloc is not allowed — and use it instead
of spec_accept. Its results must equal spec_accept's (integer outputs: bit-exact), on consecutive
calls that reuse the same scratch. This file is collected last on purpose."""
import ctypes as ct

import numpy as np
import pytest
import torch

from speculative_verify_gdn_gb300 import _lib, inputs as I

pytestmark = pytest.mark.gpu


def _static_call(lib, logits, drafts, n_acc, out, mode, temperature, seed, round_):
    d = _lib._spec_dims(logits)
    stream = ct.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.spec_accept_static(ct.byref(d), ct.c_void_p(logits.data_ptr()),
                                  ct.c_void_p(drafts.data_ptr()), int(mode),
                                  ct.c_float(temperature), int(seed), int(round_),
                                  ct.c_void_p(n_acc.data_ptr()), ct.c_void_p(out.data_ptr()),
                                  None, stream)


@pytest.mark.parametrize("mode", [_lib.SPEC_MODE_GREEDY, _lib.SPEC_MODE_SAMPLE])
def test_static_scratch_matches_workspace_entry_point(gdnlib, mode):
    lib = _lib.load()
    if mode == _lib.SPEC_MODE_GREEDY:
        w = I.WORKLOADS[1]
        temperature = 0.0
    else:
        w = I.custom(I.WORKLOADS[3], name="noalloc_sample", L=1, B=16, N=16, V=32768)
        temperature = w.temperature
    B, N = w.B, w.N
    n_ref = torch.empty(B, dtype=torch.int32, device="cuda")
    out_ref = torch.empty(B, N + 1, dtype=torch.int32, device="cuda")
    n_st = torch.empty(B, dtype=torch.int32, device="cuda")
    out_st = torch.empty(B, N + 1, dtype=torch.int32, device="cuda")
    ws = torch.empty(_lib.workspace_bytes(B, N, w.V, mode), dtype=torch.uint8, device="cuda")
    for rnd in range(2):        # two calls in a row: the second reuses the scratch left behind
        if mode == _lib.SPEC_MODE_GREEDY:
            lg, dr, _ = I.greedy_logits(w, rnd)
        else:
            lg, dr = I.sample_logits(w, rnd)
            dr[::3, ::2] = (dr[::3, ::2] + 7) % w.V
        lg, dr = lg.cuda(), dr.cuda()
        _lib.spec_accept(lg, dr, n_ref, out_ref, ws, mode=mode, temperature=temperature, seed=11,
                         round_=rnd)
        n_st.fill_(-7)
        out_st.fill_(-7)
        rc = _static_call(lib, lg, dr, n_st, out_st, mode, temperature, 11, rnd)
        assert rc == 0, _lib.last_error()
        torch.cuda.synchronize()
        assert np.array_equal(n_st.cpu().numpy(), n_ref.cpu().numpy())
        assert np.array_equal(out_st.cpu().numpy(), out_ref.cpu().numpy())


def test_static_scratch_rejects_oversized_shapes(gdnlib):
    lib = _lib.load()
    B, N, V = 400000, 1, 64      # needs more scratch than the fixed array holds
    assert _lib.workspace_bytes(B, N, V, _lib.SPEC_MODE_SAMPLE) > (1 << 20)
    lg = torch.zeros(B, N + 1, V, dtype=torch.bfloat16, device="cuda")
    dr = torch.zeros(B, N, dtype=torch.int32, device="cuda")
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, N + 1, dtype=torch.int32, device="cuda")
    rc = _static_call(lib, lg, dr, n, out, _lib.SPEC_MODE_SAMPLE, 0.7, 1, 0)
    assert rc == 2 and "static scratch" in _lib.last_error()
