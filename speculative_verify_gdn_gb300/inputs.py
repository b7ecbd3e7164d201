"""Seeded synthetic workloads for speculative verify / accept / rollback on GDN layers.

This module only draws inputs (with torch's seeded generators, on the CPU or on a CUDA device);
it holds none of the method's arithmetic and is the one piece shared by the CUDA path's tests, the
oracle's tests and the bench. Every tensor comes from a generator seeded by
(seed, workload, round, tensor name), so any piece can be regenerated independently.

Distributions (the workloads' own statements; where they are silent, the plainest reading):
  raw qkv ~ N(0, 1); beta = sigmoid(N(0, 1)); g = exp(-softplus(N(0, 1))) (per value head, or
  independently per key channel when gate_dk); S_0 ~ N(0, 0.1)
  (0.1 is the standard deviation); conv weights ~ N(0, 0.5); initial conv state ~ N(0, 1).
  Greedy logits ~ N(0, 1) with the accepted length planted; sampling logits ~ N(0, 2) with
  point-mass drafts at each row's argmax. Accept lengths are geometric: accept each position
  with probability alpha until the first miss, truncated at N, so P(n = N) = alpha^N.
"""
import zlib
from dataclasses import dataclass, field

import numpy as np
import torch

QWEN36 = dict(Hk=16, Hv=32, D=128, W=4, V=151936)


@dataclass(frozen=True)
class Workload:
    name: str
    L: int
    B: int
    N: int                      # drafts per sequence (chain) or tree nodes
    Hk: int
    Hv: int
    D: int
    W: int
    V: int
    io_dtype: torch.dtype
    accept: str                 # "greedy" | "sample" | "tree"
    alphas: tuple = (0.36,)     # per-sequence acceptance probability, cycled over b
    uniform_lengths: bool = False
    temperature: float = 0.0
    logit_std: float = 1.0
    tree_depth: int = 0
    tree_branch: int = 0
    rounds: int = 1
    gate_dk: bool = False       # one gate per key channel: g [L, B, T, Hv, D]
    notes: str = field(default="", compare=False)

    @property
    def C(self):
        return 2 * self.Hk * self.D + self.Hv * self.D

    @property
    def rows(self):
        return self.N + 1

    @property
    def P(self):
        return self.tree_depth if self.accept == "tree" else self.N


WORKLOADS = {
    0: Workload("tiny", L=1, B=1, N=4, Hk=2, Hv=4, D=32, W=4, V=1000, io_dtype=torch.float32,
                accept="greedy", uniform_lengths=True),
    1: Workload("qwen36_b1_n4", L=30, B=1, N=4, io_dtype=torch.bfloat16, accept="greedy",
                alphas=(0.36,), rounds=1, **QWEN36),
    2: Workload("qwen36_b64_n8", L=30, B=64, N=8, io_dtype=torch.bfloat16, accept="greedy",
                alphas=(0.36, 0.85), rounds=100, **QWEN36),
    3: Workload("qwen36_b16_n16_sample", L=30, B=16, N=16, io_dtype=torch.bfloat16,
                accept="sample", temperature=0.7, logit_std=2.0, **QWEN36),
    4: Workload("qwen36_b8_tree32", L=30, B=8, N=32, io_dtype=torch.bfloat16, accept="tree",
                alphas=(0.85,), tree_depth=8, tree_branch=3, **QWEN36),
}


def custom(base: Workload, **kw) -> Workload:
    d = dict(base.__dict__)
    d.update(kw)
    return Workload(**d)


_TAGS = {"conv_w": 1, "state": 2, "conv_state": 3, "qkv": 4, "g": 5, "beta": 6, "logits": 7,
         "drafts": 8, "lengths": 9, "tree": 10, "tokens": 11, "prev_delta": 12, "prev_k": 13,
         "attn_q": 14, "attn_k": 15, "attn_v": 16, "attn_kc": 17, "attn_vc": 18}

# round index of the synthetic previous round (no round loop reaches it)
PREV_ROUND = 0x7FFFFFFF


def generator(seed, wid, round_, tag, device="cpu"):
    ss = np.random.SeedSequence([int(seed), int(wid) & 0xFFFFFFFF, int(round_) & 0xFFFFFFFF,
                                 _TAGS[tag]])
    g = torch.Generator(device=device)
    g.manual_seed(int(ss.generate_state(1, dtype=np.uint64)[0] & 0x7FFFFFFFFFFFFFFF))
    return g


def _wid(w):
    """Stable id of a workload: its key in WORKLOADS, else a CRC of its name."""
    for k, v in WORKLOADS.items():
        if v.name == w.name:
            return k
    return 0x100 + (zlib.crc32(w.name.encode()) & 0xFFFFFF)


def model_weights(w: Workload, seed=0, device="cpu"):
    """conv_w [L, C, W] (io dtype)."""
    g = generator(seed, _wid(w), 0, "conv_w", device)
    cw = torch.randn((w.L, w.C, w.W), generator=g, device=device) * 0.5
    return cw.to(w.io_dtype)


def initial_state(w: Workload, seed=0, device="cpu"):
    """(state [L, B, Hv, Dv, Dk] fp32 (row-major S), conv_state [L, B, W-1, C] io dtype)."""
    g = generator(seed, _wid(w), 0, "state", device)
    st = torch.randn((w.L, w.B, w.Hv, w.D, w.D), generator=g, device=device)
    st.mul_(0.1)
    g2 = generator(seed, _wid(w), 0, "conv_state", device)
    cs = torch.randn((w.L, w.B, w.W - 1, w.C), generator=g2, device=device).to(w.io_dtype)
    return st, cs


def round_stream(w: Workload, round_, seed=0, device="cpu"):
    """Per-round verify inputs: qkv [L, B, T, C] (io), g [L, B, T, Hv] (or [L, B, T, Hv, D] when
    gate_dk), beta [L, B, T, Hv] fp32."""
    wid = _wid(w)
    T = w.N
    qkv = torch.randn((w.L, w.B, T, w.C), generator=generator(seed, wid, round_, "qkv", device),
                      device=device).to(w.io_dtype)
    gsh = (w.L, w.B, T, w.Hv) + ((w.D,) if w.gate_dk else ())
    a = torch.randn(gsh, generator=generator(seed, wid, round_, "g", device), device=device)
    g = torch.exp(-torch.nn.functional.softplus(a))
    bb = torch.randn((w.L, w.B, T, w.Hv), generator=generator(seed, wid, round_, "beta", device),
                     device=device)
    beta = torch.sigmoid(bb)
    return qkv, g.float().contiguous(), beta.float().contiguous()


def previous_round(w: Workload, seed=0, device="cpu"):
    """A synthetic previous round, the input of gdn_rollback_verify's commit half:
    (n_acc [B] int32, tape_delta [L, B, T, Hv, Dv] fp32, tape_k [L, B, T, Hk, Dk] fp32,
    g [L, B, T, Hv] fp32, qkv [L, B, T, C] io). Counts follow the workload's acceptance model;
    δ ~ N(0, 0.5); k ~ N(0, 1/D) per element (about unit length); g (of the workload's gate
    layout) and qkv as a round_stream round."""
    wid = _wid(w)
    qkv, g, _ = round_stream(w, PREV_ROUND, seed, device)
    n = accept_lengths(w, PREV_ROUND, seed, device).to(torch.int32)
    dl = torch.randn((w.L, w.B, w.N, w.Hv, w.D),
                     generator=generator(seed, wid, PREV_ROUND, "prev_delta", device), device=device)
    k = torch.randn((w.L, w.B, w.N, w.Hk, w.D),
                    generator=generator(seed, wid, PREV_ROUND, "prev_k", device), device=device)
    return n, (dl * 0.5).contiguous(), (k * (1.0 / w.D ** 0.5)).contiguous(), g, qkv


def accept_lengths(w: Workload, round_, seed=0, device="cpu"):
    """Planted accepted lengths [B] int64 (geometric per sequence, or uniform on 0..N)."""
    g = generator(seed, _wid(w), round_, "lengths", device)
    if w.uniform_lengths:
        return torch.randint(0, w.N + 1, (w.B,), generator=g, device=device)
    alpha = torch.tensor([w.alphas[b % len(w.alphas)] for b in range(w.B)], device=device)
    u = torch.rand((w.B, w.N), generator=g, device=device)
    hits = (u < alpha[:, None]).to(torch.int64)
    return torch.cumprod(hits, dim=1).sum(dim=1)


def _logit_dtype(w):
    return torch.float32 if w.io_dtype == torch.float32 else torch.bfloat16


def greedy_logits(w: Workload, round_, seed=0, device="cpu"):
    """(logits [B, N+1, V], drafts [B, N] int32, planted lengths [B]).

    Rows i < L_b get logits[b, i, d_bi] = max + 1 (strict maximum after rounding); row L_b < N has
    its draft redrawn until it differs from the row's argmax (first index among equal maxima).
    """
    wid = _wid(w)
    ldt = _logit_dtype(w)
    lg = torch.randn((w.B, w.rows, w.V), generator=generator(seed, wid, round_, "logits", device),
                     device=device).mul_(w.logit_std).to(ldt)
    gd = generator(seed, wid, round_, "drafts", device)
    drafts = torch.randint(0, w.V, (w.B, w.N), generator=gd, device=device)
    L = accept_lengths(w, round_, seed, device)
    if w.N > 0:
        rows = torch.arange(w.N, device=device)
        plant = rows[None, :] < L[:, None]                        # [B, N]
        mx = lg[:, : w.N, :].float().amax(dim=2)                  # [B, N]
        top = (mx + 1.0).to(ldt)
        bidx, iidx = plant.nonzero(as_tuple=True)
        lg[bidx, iidx, drafts[bidx, iidx]] = top[bidx, iidx]
        # row L_b (< N): draft must differ from the argmax
        am = lg[:, : w.N, :].argmax(dim=2)                       # first maximal index
        stop = rows[None, :] == L[:, None]
        clash = stop & (drafts == am)
        if clash.any():
            bidx, iidx = clash.nonzero(as_tuple=True)
            shift = torch.randint(1, w.V, (bidx.numel(),), generator=gd, device=device)
            drafts[bidx, iidx] = (am[bidx, iidx] + shift) % w.V
    return lg.contiguous(), drafts.to(torch.int32).contiguous(), L


def sample_logits(w: Workload, round_, seed=0, device="cpu"):
    """(logits [B, N+1, V] ~ N(0, logit_std), drafts = argmax of rows 0..N-1)."""
    wid = _wid(w)
    lg = torch.randn((w.B, w.rows, w.V), generator=generator(seed, wid, round_, "logits", device),
                     device=device).mul_(w.logit_std).to(_logit_dtype(w))
    drafts = lg[:, : w.N, :].argmax(dim=2).to(torch.int32)
    return lg.contiguous(), drafts.contiguous()


def random_tree(w: Workload, round_, seed=0):
    """parent [B, T] int32 (topological, -1 = child of the context) built on the CPU.

    A chain of `depth` nodes first (so the depth is exact), then each further node attaches to a
    uniformly drawn node of depth < depth with fewer than `branch` children, or to the context
    while it has fewer than `branch` children.
    """
    T, depth, br = w.N, w.tree_depth, w.tree_branch
    g = generator(seed, _wid(w), round_, "tree", "cpu")
    parents = np.full((w.B, T), -1, np.int32)
    for b in range(w.B):
        dep = np.zeros(T, np.int64)
        nchild = np.zeros(T + 1, np.int64)        # index T = the context
        for v in range(T):
            if v < min(depth, T):
                p = v - 1
            else:
                cand = [T] if nchild[T] < br else []
                cand += [u for u in range(v) if dep[u] < depth and nchild[u] < br]
                p = cand[int(torch.randint(0, len(cand), (1,), generator=g))]
                p = -1 if p == T else p
            parents[b, v] = p
            dep[v] = 1 if p < 0 else dep[p] + 1
            nchild[T if p < 0 else p] += 1
    return torch.from_numpy(parents)


def tree_tokens_and_logits(w: Workload, parent, round_, seed=0):
    """(tokens [B, T] int32 with distinct siblings, logits [B, T+1, V], planted lengths [B]).

    Row 0 judges the children of the context, row 1+v the children of node v. Along one random
    root-to-leaf path, the first L nodes (L geometric in alpha, at most the path length) are made
    the argmax of their parent's row; at the stopping node no child's token is the argmax.
    """
    wid = _wid(w)
    T = w.N
    gt = generator(seed, wid, round_, "tokens", "cpu")
    par = parent.numpy()
    tokens = np.zeros((w.B, T), np.int64)
    for b in range(w.B):
        for v in range(T):
            sib = {int(tokens[b, u]) for u in range(v) if par[b, u] == par[b, v]}
            t = int(torch.randint(0, w.V, (1,), generator=gt))
            while t in sib:
                t = int(torch.randint(0, w.V, (1,), generator=gt))
            tokens[b, v] = t
    ldt = _logit_dtype(w)
    lg = torch.randn((w.B, T + 1, w.V), generator=generator(seed, wid, round_, "logits", "cpu"))
    lg = lg.mul_(w.logit_std).to(ldt)
    gl = generator(seed, wid, round_, "lengths", "cpu")
    Ls = np.zeros(w.B, np.int64)
    for b in range(w.B):
        children = {p: [v for v in range(T) if par[b, v] == p] for p in range(-1, T)}
        leaves = [v for v in range(T) if not children[v]]
        leaf = leaves[int(torch.randint(0, len(leaves), (1,), generator=gl))]
        path = []
        x = leaf
        while x >= 0:
            path.append(x)
            x = int(par[b, x])
        path.reverse()
        alpha = w.alphas[b % len(w.alphas)]
        L = 0
        while L < len(path) and float(torch.rand((1,), generator=gl)) < alpha:
            L += 1
        Ls[b] = L
        for k in range(L):
            row = 0 if k == 0 else 1 + path[k - 1]
            lg[b, row, tokens[b, path[k]]] = (lg[b, row].float().max() + 1.0).to(ldt)
        stop = -1 if L == 0 else path[L - 1]
        row = 1 + stop
        kids = {int(tokens[b, v]) for v in children[stop]}
        for _ in range(len(kids) + 1):
            am = int(lg[b, row].argmax())
            if am not in kids:
                break
            lg[b, row, am] = (lg[b, row].float().min() - 1.0).to(ldt)
    return torch.from_numpy(tokens.astype(np.int32)), lg.contiguous(), torch.from_numpy(Ls)


# ------------------------------------------------------------------ attention layers
@dataclass(frozen=True)
class AttnWorkload:
    """The hybrid's full-attention layers in one verify step: L layers, B sequences with
    `lengths[b % len]` committed cache rows, T verify positions, Hq query heads over Hkv kv heads
    of dim D, cache capacity ctx rows."""
    name: str
    L: int
    B: int
    T: int
    Hq: int
    Hkv: int
    D: int
    ctx: int
    lengths: tuple
    notes: str = field(default="", compare=False)


# Qwen3.6-35B-A3B-shaped attention layers (10 of its 40 layers; 16 query heads over 2 kv heads of
# dim 256) over a 4096-token context, at the GDN workloads' batch and draft count.
ATTN_WORKLOADS = {
    "qwen36_attn_b64_n8": AttnWorkload("qwen36_attn_b64_n8", L=10, B=64, T=8, Hq=16, Hkv=2,
                                       D=256, ctx=4224, lengths=(4096,)),
    "qwen36_attn_b1_n8": AttnWorkload("qwen36_attn_b1_n8", L=10, B=1, T=8, Hq=16, Hkv=2, D=256,
                                      ctx=4224, lengths=(4096,)),
    "qwen36_attn_b16_n16": AttnWorkload("qwen36_attn_b16_n16", L=10, B=16, T=16, Hq=16, Hkv=2,
                                        D=256, ctx=4224, lengths=(4096,)),
}


def _awid(w):
    return 0x200 + (zlib.crc32(w.name.encode()) & 0xFFFFFF)


def attn_lengths(w: AttnWorkload):
    """Committed cache rows per sequence, int32 [B]."""
    return torch.tensor([w.lengths[b % len(w.lengths)] for b in range(w.B)], dtype=torch.int32)


def attn_round(w: AttnWorkload, round_, seed=0, device="cpu"):
    """One verify step's projected q [L, B, T, Hq, D] and new k, v [L, B, T, Hkv, D], bf16,
    every element N(0, 1)."""
    wid = _awid(w)
    out = []
    for tag, h in (("attn_q", w.Hq), ("attn_k", w.Hkv), ("attn_v", w.Hkv)):
        t = torch.randn((w.L, w.B, w.T, h, w.D), generator=generator(seed, wid, round_, tag, device),
                        device=device)
        out.append(t.to(torch.bfloat16))
    return tuple(out)


def attn_cache(w: AttnWorkload, seed=0, device="cpu"):
    """(k_cache, v_cache) [L, B, Hkv, ctx, D] bf16, token-major: rows below each sequence's
    committed length ~ N(0, 1), the rest zero (allocated zeroed, as a cache is)."""
    wid = _awid(w)
    kc = torch.randn((w.L, w.B, w.Hkv, w.ctx, w.D), generator=generator(seed, wid, 0, "attn_kc", device),
                     device=device).to(torch.bfloat16)
    vc = torch.randn((w.L, w.B, w.Hkv, w.ctx, w.D), generator=generator(seed, wid, 0, "attn_vc", device),
                     device=device).to(torch.bfloat16)
    n = attn_lengths(w).to(device)
    keep = (torch.arange(w.ctx, device=device)[None, :] < n[:, None].long())   # [B, ctx]
    m = keep[None, :, None, :, None]
    return kc * m, vc * m

