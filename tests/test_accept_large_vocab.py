"""Greedy and tree accept at model-sized vocabularies (8192 to 262147, bf16 and fp32 logits, rows
padded to a 16-byte stride): token ids, counts and paths bit-exact with the oracle, over ragged
batches, ties across the vocabulary chunks, NaN logits, deep accept runs, zero drafts, bad drafts /
parents, and path capacities below the tree's depth."""
import numpy as np
import pytest
import torch

import oracle
from speculative_verify_gdn_gb300 import _lib, inputs as I
from parity_util import logits_f32, to_dev

pytestmark = pytest.mark.gpu


def padded(lg, dtype):
    """Rows padded to a 16-byte stride with values that must never be read."""
    VN = 8 if dtype == torch.bfloat16 else 4
    B, R, V = lg.shape
    Vpad = (V + VN - 1) // VN * VN
    pad = torch.full((B, R, Vpad), 1e4).to(dtype)
    pad[..., :V] = lg.to(dtype)
    return pad


def greedy_case(B, N, V, dtype, seed, plant=None, std=2.0, rounds=2):
    g = np.random.default_rng(seed)
    ws = torch.empty(_lib.workspace_bytes(B, N, V, _lib.SPEC_MODE_GREEDY, dtype), dtype=torch.uint8,
                     device="cuda")
    n_acc = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, N + 1, dtype=torch.int32, device="cuda")
    ns = []
    for _ in range(rounds):
        lg = torch.from_numpy((g.standard_normal((B, N + 1, V)) * std).astype(np.float32))
        lg = lg.to(dtype).float()
        dr = lg[:, :N].argmax(-1).to(torch.int32)         # every draft right ...
        for b in range(B):                                # ... up to a random first miss
            stop = int(g.integers(0, N + 2))
            if stop < N:
                dr[b, stop] = (dr[b, stop] + 1 + int(g.integers(0, V - 1))) % V
        if plant is not None:
            plant(lg, dr, g)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        dlg, ddr = to_dev(padded(lg, dtype), dr)
        _lib.spec_accept(dlg, ddr, n_acc, out, ws, mode=_lib.SPEC_MODE_GREEDY, status=status, V=V)
        torch.cuda.synchronize()
        n, out_ref, bad = oracle.accept_greedy(logits_f32(lg.to(dtype)), dr.numpy())
        assert np.array_equal(n_acc.cpu().numpy(), n)
        assert np.array_equal(out.cpu().numpy(), out_ref)
        assert (int(status.item()) != 0) == (bad != 0)
        ns.append(n)
    return np.concatenate(ns)


@pytest.mark.parametrize("V,dtype,B", [(8192, torch.bfloat16, 5), (8193, torch.float32, 3),
                                       (50001, torch.bfloat16, 37), (151936, torch.bfloat16, 64),
                                       (151936, torch.float32, 7), (262147, torch.bfloat16, 4),
                                       (163841, torch.float32, 2)])
def test_greedy_accept_vocab_sizes(gdnlib, V, dtype, B):
    n = greedy_case(B, 8, V, dtype, seed=V % 89 + B)
    assert n.min() < 8 and n.max() > 0


def test_greedy_accept_ties_and_nan(gdnlib):
    """Equal maxima in different vocabulary chunks (the lowest index wins), NaN logits (never picked;
    a NaN / −∞ row gives index 0), the maximum at the very last token."""
    B, N, V = 6, 4, 151936

    def plant(lg, dr, g):
        nan, inf = float("nan"), float("inf")
        lg[0, 0, 100] = lg[0, 0, 140000] = 50.0          # tie across chunks: 100 wins
        dr[0, 0] = 100
        lg[1, 1, V - 1] = 60.0                            # last token
        dr[1, 0] = int(lg[1, 0].argmax())
        dr[1, 1] = V - 1
        lg[2, 0, :] = nan                                 # a NaN row: index 0
        dr[2, 0] = 0
        lg[3, 2, :] = -inf
        lg[3, 2, 70000:] = nan                            # −∞ and NaN: index 0
        lg[4, 0, int(lg[4, 0].argmax())] = nan            # the maximum becomes NaN
        lg[5, :, 151000:] = nan

    greedy_case(B, N, V, torch.float32, seed=3, plant=plant, rounds=1)


def test_greedy_accept_every_draft_and_zero_drafts(gdnlib):
    """All drafts right (the bonus row is reached), and N = 0 (only the bonus row)."""
    def allright(lg, dr, g):
        dr[:] = lg[:, :dr.shape[1]].argmax(-1).to(torch.int32)

    n = greedy_case(9, 16, 151936, torch.bfloat16, seed=4, plant=allright, rounds=1)
    assert (n == 16).all()
    greedy_case(9, 0, 151936, torch.bfloat16, seed=5, rounds=2)


def test_greedy_accept_bad_draft_large_vocab(gdnlib):
    B, N, V = 5, 6, 151936

    def plant(lg, dr, g):
        dr[1, 4] = V
        dr[3, 0] = -2

    greedy_case(B, N, V, torch.bfloat16, seed=6, plant=plant, rounds=1)


def tree_accept_case(B, T, V, dtype, depth, branch, P, seed, edit=None):
    w = I.custom(I.WORKLOADS[4], name="tree_acc_%d_%d_%d" % (B, T, V), B=B, N=T, V=V,
                 tree_depth=depth, tree_branch=branch, io_dtype=dtype)
    par = I.random_tree(w, 0, seed)
    tok, lg, _ = I.tree_tokens_and_logits(w, par, 0, seed)
    if edit is not None:
        edit(par, tok, lg)
    lg = lg.to(dtype)
    ws = torch.empty(_lib.workspace_bytes(B, T, V, _lib.SPEC_MODE_GREEDY, dtype), dtype=torch.uint8,
                     device="cuda")
    path = torch.empty(B, P, dtype=torch.int32, device="cuda")
    n_acc = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, P + 1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dlg, dpar, dtok = to_dev(padded(lg.float(), dtype), par, tok)
    _lib.spec_accept_tree(dlg, dpar, dtok, path, n_acc, out, ws, status=status, V=V)
    torch.cuda.synchronize()
    path_ref, n, out_ref, bad = oracle.accept_tree(logits_f32(lg), par.numpy(), tok.numpy(), P)
    assert np.array_equal(n_acc.cpu().numpy(), n)
    assert np.array_equal(path.cpu().numpy(), path_ref)
    assert np.array_equal(out.cpu().numpy(), out_ref)
    assert (int(status.item()) != 0) == (bad != 0)
    return n, int(status.item())


@pytest.mark.parametrize("B,T,V,dtype,depth,branch,P", [
    (8, 32, 151936, torch.bfloat16, 8, 3, 8),           # the benchmarked tree shape
    (5, 32, 151936, torch.bfloat16, 8, 3, 4),           # path capacity below the depth
    (3, 17, 8192, torch.float32, 5, 2, 17),
    (21, 12, 50001, torch.bfloat16, 12, 1, 12),         # one chain
    (4, 24, 131073, torch.float32, 2, 24, 2),           # a bush: many children per node
])
def test_tree_accept_large_vocab(gdnlib, B, T, V, dtype, depth, branch, P):
    tree_accept_case(B, T, V, dtype, depth, branch, P, seed=T + B)


def test_tree_accept_bad_parent_and_token_large_vocab(gdnlib):
    def edit(par, tok, lg):
        par[1, 5] = 7                                     # not topological
        tok[2, 3] = 151936                                # outside the vocabulary

    n, st = tree_accept_case(4, 16, 151936, torch.bfloat16, 6, 3, 6, seed=2, edit=edit)
    assert st & 0x2 and st & 0x4                     # BAD_PARENT, BAD_TOKEN
    assert n[1] == 0 and n[2] == 0
