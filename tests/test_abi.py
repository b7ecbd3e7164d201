"""The C-ABI library builds, loads without a GPU, exports every entry point include/*.h declares,
and its host-side checks (sizes, argument validation) work with no device. No compute calls."""
import ctypes as ct
import glob
import os
import re

import pytest

from speculative_verify_gdn_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"GDN_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_header_declares_the_expected_calls():
    assert set(declared_functions()) == set(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_no_unexpected_exports(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.library_path()], capture_output=True,
                         text=True).stdout
    syms = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    extra = {s for s in syms if not s.startswith("_")} - set(_lib.EXPORTS)
    assert not extra, extra


def qwen_shape(**kw):
    d = dict(L=30, B=64, T=8, Hk=16, Hv=32, Dk=128, Dv=128, W=4)
    d.update(kw)
    return _lib.GdnShape(**d)


def test_tape_bytes(lib):
    sh = qwen_shape()
    expect = 30 * 64 * 8 * (32 * 128 + 16 * 128) * 4
    assert _lib.tape_bytes(sh) == expect
    assert _lib.tape_bytes(qwen_shape(Dk=96, Dv=96)) == 0       # unsupported head dim
    assert _lib.tape_bytes(qwen_shape(Hv=24)) == 0             # Hv not a multiple of Hk... 24%16


def test_workspace_bytes(lib):
    g = _lib.workspace_bytes(64, 8, 151936)
    s = _lib.workspace_bytes(64, 8, 151936, _lib.SPEC_MODE_SAMPLE)
    assert g > 0 and s > 2 * g - 1
    assert _lib.workspace_bytes(1, 4, 151936) >= 5 * 8


def call_verify(lib, d, ptrs):
    return lib.gdn_verify(ct.byref(d), *ptrs, None, None)


def test_host_validation_rejects_bad_arguments_without_a_gpu(lib):
    fake = ct.c_void_p(0x100000)        # never dereferenced: validation fails first
    d = qwen_shape().c()
    # NULL tensors
    assert call_verify(lib, d, [None] * 9) == 1
    assert "NULL" in _lib.last_error()
    # inconsistent channel count
    d2 = qwen_shape().c()
    d2.C = 100
    assert call_verify(lib, d2, [fake] * 9) == 1
    assert "C=" in _lib.last_error()
    # unsupported head dim / conv width / T
    assert call_verify(lib, qwen_shape(Dk=96, Dv=96).c(), [fake] * 9) == 2
    assert call_verify(lib, qwen_shape(W=5).c(), [fake] * 9) == 2
    assert call_verify(lib, qwen_shape(T=33).c(), [fake] * 9) == 2
    # misaligned state
    bad = [fake] * 9
    bad[5] = ct.c_void_p(0x100004)
    assert call_verify(lib, d, bad) == 1 and "aligned" in _lib.last_error()
    # empty shapes are no-ops (no launch)
    assert call_verify(lib, qwen_shape(B=0).c(), [None] * 9) == 0
    # rollback / accept argument checks
    assert lib.gdn_rollback(ct.byref(d), None, None, None, None, None, None, None, None,
                            None) == 1
    sd = _lib._SpecDims(4, 3, 1000, _lib.GDN_DTYPE_BF16, 1001, 0)    # stride not 16-byte
    assert lib.spec_accept(ct.byref(sd), fake, fake, 0, 0.0, 0, 0, fake, 1 << 20, fake, fake,
                           None, None) == 1
    sd = _lib._SpecDims(4, 3, 1000, _lib.GDN_DTYPE_BF16, 1000, 4000)
    assert lib.spec_accept(ct.byref(sd), fake, fake, 0, 0.0, 0, 0, fake, 8, fake, fake,
                           None, None) == 1
    assert "workspace" in _lib.last_error()
    assert lib.spec_accept(ct.byref(sd), fake, fake, 7, 0.0, 0, 0, fake, 1 << 20, fake, fake,
                           None, None) == 1
    # tree accept: at most 4096 nodes (the walk stages parents and tokens in shared memory)
    td = _lib._SpecDims(2, 4097, 1000, _lib.GDN_DTYPE_BF16, 1000, 4098 * 1000)
    assert lib.spec_accept_tree(ct.byref(td), fake, fake, fake, 8, fake, 1 << 30, fake, fake,
                                fake, None, None) == 2
    assert "4096" in _lib.last_error()


def test_rollback_verify_host_checks(lib):
    d = qwen_shape().c()
    # distinct, non-overlapping, never dereferenced (validation fails before any CUDA call)
    args = [ct.c_void_p((i + 1) << 32) for i in range(15)]   # n_acc_prev .. tape_k
    assert lib.gdn_rollback_verify(ct.byref(d), *([None] * 15), None, None) == 1
    assert "NULL" in _lib.last_error()
    # this round's tape on top of the previous round's tape
    same = list(args)
    same[1] = ct.c_void_p(0x200000)     # tape_delta_prev
    same[13] = ct.c_void_p(0x200000)    # tape_delta
    assert lib.gdn_rollback_verify(ct.byref(d), *same, None, None) == 1
    assert "overlap" in _lib.last_error()
    # misaligned previous tape (bulk copies need 16 bytes)
    mis = list(args)
    mis[2] = ct.c_void_p(0x300004)      # tape_k_prev
    assert lib.gdn_rollback_verify(ct.byref(d), *mis, None, None) == 1
    assert "aligned" in _lib.last_error()
    assert lib.gdn_rollback_verify(ct.byref(qwen_shape(B=0).c()), *([None] * 15), None, None) == 0


def test_struct_layouts_match_the_header(tmp_path):
    """gdn_dims / spec_dims as the C compiler lays them out equal the ctypes mirrors in _lib."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = {"gdn_dims": [f for f, _ in _lib._Dims._fields_],
              "spec_dims": [f for f, _ in _lib._SpecDims._fields_],
              "attn_dims": [f for f, _ in _lib._AttnDims._fields_]}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "gdnspec.h"', "int main(void) {"]
    for st, fs in fields.items():
        lines.append('printf("%s %%zu\\n", sizeof(%s));' % (st, st))
        for f in fs:
            lines.append('printf("%s.%s %%zu\\n", offsetof(%s, %s));' % (st, f, st, f))
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = dict(l.split() for l in subprocess.run([str(exe)], check=True, capture_output=True,
                                                  text=True).stdout.splitlines())
    for st, cls in (("gdn_dims", _lib._Dims), ("spec_dims", _lib._SpecDims),
                    ("attn_dims", _lib._AttnDims)):
        assert int(got[st]) == ct.sizeof(cls), st
        for f in fields[st]:
            assert int(got["%s.%s" % (st, f)]) == getattr(cls, f).offset, (st, f)


def test_gate_dk_host_checks(lib):
    """Per-key-channel gates: fp32 trees at d = 128 are limited to 16 nodes, other values of the
    flag are rejected, all before any device access."""
    import torch
    fake = ct.c_void_p(0x100000)
    d = qwen_shape(T=32, io_dtype=torch.float32).c()
    d.gate_dk = 1
    assert lib.gdn_verify_tree(ct.byref(d), fake, *([fake] * 9), None, None) == 2
    assert "gate" in _lib.last_error()
    d.gate_dk = 2
    assert call_verify(lib, d, [fake] * 9) == 1 and "gate_dk" in _lib.last_error()


def test_attn_host_checks(lib):
    """attn_verify / attn_truncate argument checks and the workspace size, with no device."""
    fake = ct.c_void_p(0x100000)
    sh = _lib.AttnShape(L=10, B=64, T=8, Hq=16, Hkv=2, D=256, ctx=4224)
    d = sh.c()
    call = lambda dd, ptrs, ws=None, nws=0: lib.attn_verify(ct.byref(dd), *ptrs, ws, nws, None,
                                                            None)
    assert call(d, [None] * 7) == 1 and "NULL" in _lib.last_error()
    # 1280 units: 1216 run whole (8 waves over 152 SMs), the 64 left over as 2 key ranges each,
    # whose partials (64 query rows of D + 2 floats) go through the workspace
    assert lib.attn_workspace_bytes(ct.byref(d)) == 2 * 64 * 64 * (256 + 2) * 4
    whole = _lib.AttnShape(L=4, B=19, T=8, Hq=16, Hkv=2, D=256, ctx=4224)     # 152 units
    assert _lib.attn_workspace_bytes(whole) == 0
    small = _lib.AttnShape(L=1, B=1, T=8, Hq=16, Hkv=2, D=256, ctx=4224)
    assert _lib.attn_workspace_bytes(small) > 0
    # the split case needs its workspace
    assert call(small.c(), [fake] * 7) == 1 and "workspace" in _lib.last_error()
    for bad, code in ((dict(D=64), 2), (dict(T=17), 2), (dict(ctx=100), 2), (dict(ctx=4160), 2),
                      (dict(Hq=15), 1), (dict(Hkv=0), 1)):
        kw = dict(sh.__dict__)
        kw.update(bad)
        assert call(_lib.AttnShape(**kw).c(), [fake] * 7) == code, bad
    mis = [fake] * 7
    mis[3] = ct.c_void_p(0x100008)            # k_cache not 16-byte aligned
    assert call(d, mis) == 1 and "aligned" in _lib.last_error()
    assert call(_lib.AttnShape(L=10, B=0, T=8, Hq=16, Hkv=2, D=256, ctx=4224).c(),
                [None] * 7) == 0
    assert lib.attn_truncate(4, 8, None, None, None, None) == 1
    assert lib.attn_truncate(0, 8, None, None, None, None) == 0



def test_value_cache_tile_layout():
    """The tile-transposed value cache: position j, dim d sits at [j // 128, d, j % 128]."""
    import torch
    v = torch.randn(2, 3, 256, 16)
    vt = _lib.vt_from_v(v)
    assert vt.shape == (2, 3, 2, 16, 128) and vt.is_contiguous()
    for j in (0, 5, 127, 128, 200, 255):
        for d in (0, 7, 15):
            assert vt[1, 2, j // 128, d, j % 128] == v[1, 2, j, d]
    assert torch.equal(_lib.v_from_vt(vt), v)


def test_status_check_maps_device_bits_to_an_error(lib):
    assert lib.gdn_status_check(0) == _lib.GDN_OK
    assert lib.gdn_status_check(0x1 | 0x20) == _lib.GDN_ERR_DEVICE_STATUS
    msg = _lib.last_error()
    assert "BAD_NACC" in msg and "WAIT_TIMEOUT" in msg and "BAD_TOKEN" not in msg
    assert lib.gdn_status_check(0x80000000) == _lib.GDN_ERR_DEVICE_STATUS
    assert "unknown bits 0x80000000" in _lib.last_error()
    with pytest.raises(_lib.GdnError, match="BAD_PATH"):
        _lib.status_check(0x8)
    _lib.status_check(0)
