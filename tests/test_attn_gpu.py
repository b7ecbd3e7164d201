"""GPU parity of the attention-layer verify (attn_verify: KV-cache append + causal GQA attention
of the T verify positions) and the KV truncation (attn_truncate) against the oracle, on seeded
synthetic inputs.

Tolerance for o (derived from the arithmetic): the kernel rounds each softmax weight to bf16 (8
significant bits) for the tensor core and normalises by the sum of the rounded weights, so every
normalised weight carries a relative error below 2^-8 and
    |gpu - ref| <= 2^-8 · Σ_j p_j |v_j| + 1e-5 · max|ref| + ulp_bf16(ref) / 2,
with Σ_j p_j |v_j| taken from the oracle run on |v|. The appended cache rows and the lengths are
compared bit-exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import AttnDims
from speculative_verify_gdn_gb300 import _lib, inputs as I
from parity_util import half_ulp_bf16

pytestmark = pytest.mark.gpu


def f64(t):
    return t.detach().to("cpu").double().numpy()


def workload(L=2, B=3, T=4, Hq=4, Hkv=2, D=128, ctx=384, lengths=(0, 130, 300)):
    name = "attn_L%d_B%d_T%d_H%d_%d_D%d_c%d_%s" % (L, B, T, Hq, Hkv, D, ctx,
                                                   "_".join(map(str, lengths)))
    return I.AttnWorkload(name, L=L, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, ctx=ctx, lengths=lengths)


def shape_of(w):
    return _lib.AttnShape(L=w.L, B=w.B, T=w.T, Hq=w.Hq, Hkv=w.Hkv, D=w.D, ctx=w.ctx)


def run_gpu(w, q, kn, vn, kc, vc, kv_len, status=None, out_fill=None):
    sh = shape_of(w)
    dq, dkn, dvn = q.cuda(), kn.cuda(), vn.cuda()
    dkc = kc.cuda().contiguous()
    dvt = _lib.vt_from_v(vc).cuda()                         # the tile-transposed value cache
    dlen = kv_len.cuda()
    out = torch.zeros(sh.q_shape(), dtype=torch.bfloat16, device="cuda")
    if out_fill is not None:
        out.fill_(out_fill)
    nws = _lib.attn_workspace_bytes(sh)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda") if nws else None
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.attn_verify(sh, dq, dkn, dvn, dkc, dvt, dlen, out, workspace=ws, status=status)
    torch.cuda.synchronize()
    return out, dkc, dvt, dlen, status


def run_oracle(w, q, kn, vn, kc, vc, kv_len):
    d = AttnDims(L=w.L, B=w.B, T=w.T, Hq=w.Hq, Hkv=w.Hkv, D=w.D, ctx=w.ctx,
                 scale=float(np.float32(1.0 / np.sqrt(w.D))))
    out, kc2, vc2, bad = oracle.attn_verify(d, kv_len.numpy(), f64(q), f64(kn), f64(vn), f64(kc),
                                            f64(vc))
    absout, _, _, _ = oracle.attn_verify(d, kv_len.numpy(), f64(q), f64(kn), np.abs(f64(vn)),
                                         f64(kc), np.abs(f64(vc)))
    return out, absout, kc2, vc2, bad


def assert_attn_close(gpu, ref, ref_abs, name="out"):
    gpu = np.asarray(gpu, np.float64)
    bound = 2.0 ** -8 * ref_abs + 1e-5 * np.abs(ref).max() + half_ulp_bf16(ref)
    err = np.abs(gpu - ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), ref.shape)
        raise AssertionError("%s: %d/%d out of tolerance; worst at %s: gpu=%r ref=%r bound=%r"
                             % (name, bad.sum(), bad.size, i, gpu[i], ref[i], bound[i]))


def check_case(w, seed=0):
    q, kn, vn = I.attn_round(w, 0, seed)
    kc, vc = I.attn_cache(w, seed)
    kv_len = I.attn_lengths(w)
    out, dkc, dvt, dlen, status = run_gpu(w, q, kn, vn, kc, vc, kv_len)
    assert int(status.item()) == 0, _lib.decode_status(int(status.item()))
    ref, ref_abs, kc2, vc2, bad = run_oracle(w, q, kn, vn, kc, vc, kv_len)
    assert bad == 0
    assert_attn_close(f64(out), ref, ref_abs)
    # the append: bit-exact, and nothing else written
    assert np.array_equal(f64(dkc), kc2)
    assert np.array_equal(f64(_lib.v_from_vt(dvt)), vc2)
    assert torch.equal(dlen.cpu(), kv_len)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("T,Hq,Hkv", [(1, 4, 2), (4, 4, 2), (8, 16, 2), (3, 8, 8), (16, 16, 2),
                                      (5, 6, 2)])
def test_attn_matches_oracle(gdnlib, D, T, Hq, Hkv):
    """Ragged cache lengths (empty, one row past a tile, mid-tile), every query-row padding."""
    check_case(workload(T=T, Hq=Hq, Hkv=Hkv, D=D), seed=T + Hq)


@pytest.mark.parametrize("ctx,lengths", [(128, (0, 120, 64)), (1024, (1000, 7, 511)),
                                         (256, (248, 0, 1))])
def test_attn_cache_edges(gdnlib, ctx, lengths):
    """Capacity exactly one tile, the last rows of the cache (full capacity after the append)."""
    check_case(workload(T=8, Hq=16, Hkv=2, D=256, ctx=ctx, lengths=lengths), seed=ctx)


def test_attn_split_keys(gdnlib):
    """Few (layer, sequence, kv head) units over a long cache: the keys are split across CTAs
    and merged by the combine kernel."""
    w = workload(L=1, B=1, T=8, Hq=16, Hkv=2, D=256, ctx=2048, lengths=(2000,))
    sh = shape_of(w)
    assert _lib.attn_workspace_bytes(sh) > 0
    check_case(w, seed=11)


@pytest.mark.parametrize("ctx,lengths,L,B", [(2048, (2000,), 1, 1), (128, (0, 112, 57), 2, 3),
                                             (640, (600, 1, 128), 1, 3)])
def test_attn_128_query_rows(gdnlib, ctx, lengths, L, B):
    """T = 16 over 8 query heads per kv head: 128 query rows per kv head, run as two 64-row CTAs
    of one cluster sharing every K / V load; with the keys split across CTAs (first case), an
    empty cache, a cache filled to capacity by the append, and one key."""
    check_case(workload(L=L, B=B, T=16, Hq=16, Hkv=2, D=256, ctx=ctx, lengths=lengths),
               seed=ctx + B)


@pytest.mark.parametrize("T", [8, 16])
def test_attn_whole_and_split_units_in_one_call(gdnlib, T):
    """154 units: 152 run whole (one wave over 152 SMs), the 2 left over as key ranges whose
    partials the combine kernel merges; both kernels (64 and 128 query rows), ragged lengths."""
    w = workload(L=1, B=77, T=T, Hq=16, Hkv=2, D=128, ctx=512,
                 lengths=(0, 300, 512 - T, 129, 77, 200, 1))
    assert _lib.attn_workspace_bytes(shape_of(w)) > 0
    check_case(w, seed=T)


def test_attn_large_scores_stay_finite(gdnlib):
    """Scores of a few hundred (q and k scaled up): the running maximum moves by large steps and
    the rescaling of O must keep everything finite and exact to the tolerance."""
    w = workload(L=1, B=2, T=8, Hq=16, Hkv=2, D=128, ctx=640, lengths=(600, 200))
    q, kn, vn = I.attn_round(w, 0, 5)
    kc, vc = I.attn_cache(w, 5)
    q = (q.float() * 6).to(torch.bfloat16)
    kn = (kn.float() * 3).to(torch.bfloat16)
    kc = (kc.float() * 3).to(torch.bfloat16)
    kv_len = I.attn_lengths(w)
    out, _, _, _, status = run_gpu(w, q, kn, vn, kc, vc, kv_len)
    assert int(status.item()) == 0
    ref, ref_abs, _, _, _ = run_oracle(w, q, kn, vn, kc, vc, kv_len)
    assert np.isfinite(f64(out)).all()
    assert_attn_close(f64(out), ref, ref_abs)


def test_attn_misaligned_new_values_are_rejected(gdnlib):
    """v_new is read in 16-byte pieces: a pointer off that boundary is refused before any launch,
    and nothing is written."""
    w = workload(L=1, B=1, T=4, Hq=4, Hkv=2, D=128, ctx=256, lengths=(10,))
    sh = shape_of(w)
    q, kn, vn = [t.cuda() for t in I.attn_round(w, 0, 1)]
    kc, vc = I.attn_cache(w, 1)
    dkc, dvt = kc.cuda(), _lib.vt_from_v(vc).cuda()
    vbuf = torch.zeros(vn.numel() + 8, dtype=torch.bfloat16, device="cuda")
    vshift = vbuf[1:1 + vn.numel()].view(vn.shape)          # 2 bytes past a 16-byte boundary
    vshift.copy_(vn)
    out = torch.full(sh.q_shape(), 7.0, dtype=torch.bfloat16, device="cuda")
    before = dkc.clone()
    with pytest.raises(_lib.GdnError, match="16-byte"):
        _lib.attn_verify(sh, q, kn, vshift, dkc, dvt, torch.tensor([10], dtype=torch.int32,
                                                                 device="cuda"), out)
    torch.cuda.synchronize()
    assert torch.equal(dkc, before) and bool((out == 7.0).all())


def test_attn_bad_length_is_reported_and_skipped(gdnlib):
    w = workload(L=1, B=2, T=4, Hq=4, Hkv=2, D=128, ctx=256, lengths=(100, 100))
    q, kn, vn = I.attn_round(w, 0, 1)
    kc, vc = I.attn_cache(w, 1)
    kv_len = torch.tensor([253, 100], dtype=torch.int32)        # 253 + 4 > 256
    out, dkc, _, _, status = run_gpu(w, q, kn, vn, kc, vc, kv_len, out_fill=7.0)
    assert int(status.item()) & 0x40
    assert (out[:, 0] == 7.0).all() and torch.equal(dkc[:, 0].cpu(), kc[:, 0])
    ref, ref_abs, _, _, bad = run_oracle(w, q, kn, vn, kc, vc, kv_len)
    assert bad == 1
    assert_attn_close(f64(out[:, 1:]), ref[:, 1:], ref_abs[:, 1:])


def test_attn_truncate_matches_oracle(gdnlib):
    n = torch.tensor([0, 8, 3, 9, -1, 5], dtype=torch.int32)
    kl = torch.tensor([100, 200, 300, 400, 500, 0], dtype=torch.int32)
    dn, dkl = n.cuda(), kl.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.attn_truncate(dn, dkl, 8, status=st)
    torch.cuda.synchronize()
    ref, bad = oracle.attn_truncate(8, n.numpy(), kl.numpy())
    assert bad == 1 and int(st.item()) & 0x1
    assert dkl.cpu().numpy().tolist() == ref.tolist()


def test_attn_round_trip_append_truncate_append(gdnlib):
    """Two rounds: append + attend, truncate to the accepted counts, then the next round's rows
    land right after the kept ones (the rejected rows are overwritten)."""
    w = workload(L=1, B=3, T=4, Hq=8, Hkv=2, D=128, ctx=256, lengths=(10, 50, 0))
    q, kn, vn = I.attn_round(w, 0, 2)
    kc, vc = I.attn_cache(w, 2)
    kv_len = I.attn_lengths(w)
    _, dkc, dvt, dlen, status = run_gpu(w, q, kn, vn, kc, vc, kv_len)
    n_acc = torch.tensor([1, 4, 0], dtype=torch.int32)
    _lib.attn_truncate(n_acc.cuda(), dlen, w.T, status=status)
    q2, kn2, vn2 = I.attn_round(w, 1, 2)
    sh = shape_of(w)
    out2 = torch.empty(sh.q_shape(), dtype=torch.bfloat16, device="cuda")
    nws = _lib.attn_workspace_bytes(sh)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda") if nws else None
    _lib.attn_verify(sh, q2.cuda(), kn2.cuda(), vn2.cuda(), dkc, dvt, dlen, out2, workspace=ws,
                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # oracle: the same two rounds
    _, _, kc1, vc1, _ = run_oracle(w, q, kn, vn, kc, vc, kv_len)
    kl1, _ = oracle.attn_truncate(w.T, n_acc.numpy(), kv_len.numpy())
    assert dlen.cpu().numpy().tolist() == kl1.tolist()
    ref2, ref2_abs, kc2, vc2, _ = run_oracle(w, q2, kn2, vn2, torch.from_numpy(kc1),
                                             torch.from_numpy(vc1), torch.from_numpy(kl1))
    assert_attn_close(f64(out2), ref2, ref2_abs)
    assert np.array_equal(f64(dkc), kc2)
    assert np.array_equal(f64(_lib.v_from_vt(dvt)), vc2)


@pytest.mark.parametrize("name", ["qwen36_attn_b64_n8", "qwen36_attn_b16_n16"])
def test_attn_full_size_sampled_units(gdnlib, name):
    """The benchmarked workloads (10 layers, 4096 committed rows, 16 query heads over 2 kv heads
    of dim 256; batch 64 at T = 8, batch 16 at T = 16), inputs drawn on the device; two (layer,
    sequence) units compared with the oracle, and every output finite."""
    w = I.ATTN_WORKLOADS[name]
    dev = "cuda"
    q, kn, vn = I.attn_round(w, 0, 0, dev)
    kc, vc = I.attn_cache(w, 0, dev)
    vt = _lib.vt_from_v(vc)
    kv_len = I.attn_lengths(w).to(dev)
    sh = shape_of(w)
    out = torch.empty(sh.q_shape(), dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    kc_before = {}
    units = [(0, 0), (7, min(41, w.B - 1)), (w.L - 1, w.B - 1)]   # the last: a key-split tail unit
    for (l, b) in units:
        kc_before[(l, b)] = (kc[l, b].clone(), vc[l, b].clone())
    nws = _lib.attn_workspace_bytes(sh)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev) if nws else None
    _lib.attn_verify(sh, q, kn, vn, kc, vt, kv_len, out, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.isfinite(out.float()).all()
    one = I.AttnWorkload("one", L=1, B=1, T=w.T, Hq=w.Hq, Hkv=w.Hkv, D=w.D, ctx=w.ctx,
                         lengths=(w.lengths[0],))
    for (l, b) in units:
        k0, v0 = kc_before[(l, b)]
        ref, ref_abs, _, _, bad = run_oracle(
            one, q[l:l + 1, b:b + 1].cpu(), kn[l:l + 1, b:b + 1].cpu(), vn[l:l + 1, b:b + 1].cpu(),
            k0[None, None].cpu(), v0[None, None].cpu(), kv_len[b:b + 1].cpu())
        assert bad == 0
        assert_attn_close(f64(out[l:l + 1, b:b + 1]), ref, ref_abs, "out unit %s" % ((l, b),))
