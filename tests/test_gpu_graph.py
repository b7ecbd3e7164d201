"""Speculative rounds captured in a CUDA graph: the library only enqueues work on the caller's
stream (no allocation, no synchronisation, host-side plans made on first use), so a round loop of
verify -> accept -> rollback can be captured once and replayed. The replay must give the same
accepted counts, tokens, state and conv state, bit for bit, as the same calls made eagerly."""
import pytest
import torch

from speculative_verify_gdn_gb300 import inputs as I
from speculative_verify_gdn_gb300.round import SpecRound

pytestmark = pytest.mark.gpu


def round_inputs(w, k, device="cuda"):
    qkv, g, beta = I.round_stream(w, k, 0, device)
    if w.accept == "sample":
        lg, dr = I.sample_logits(w, k, 0, device)
    else:
        lg, dr, _ = I.greedy_logits(w, k, 0, device)
    return dict(qkv=qkv, g=g, beta=beta, logits=lg, drafts=dr)


@pytest.mark.parametrize("kind", ["greedy", "sample"])
def test_round_loop_replays_from_a_cuda_graph(gdnlib, kind):
    base = I.WORKLOADS[2] if kind == "greedy" else I.WORKLOADS[3]
    w = I.custom(base, name="graph_" + kind, L=3, B=6, N=8, V=16384)
    rounds = 3
    cw = I.model_weights(w, 0, "cuda")
    st0, cs0 = I.initial_state(w, 0, "cuda")
    ins = [round_inputs(w, k) for k in range(rounds)]

    def run(r, st, cs, logs):
        for k in range(rounds):
            s = ins[k]
            r.step(s["qkv"], s["g"], s["beta"], s["logits"], s["drafts"], cw, st, cs, round_=k,
                   seed=11)
            logs[k][0].copy_(r.n_acc)
            logs[k][1].copy_(r.out_tokens)

    def logs_for(r):
        return [(torch.empty_like(r.n_acc), torch.empty_like(r.out_tokens)) for _ in range(rounds)]

    # eager
    r_e = SpecRound(w)
    st_e, cs_e = st0.clone(), cs0.clone()
    log_e = logs_for(r_e)
    run(r_e, st_e, cs_e, log_e)
    r_e.check_status()

    # captured once (after a warm-up that makes the library's first-use plans), then replayed
    r_g = SpecRound(w)
    st_g, cs_g = st0.clone(), cs0.clone()
    log_g = logs_for(r_g)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run(r_g, st_g, cs_g, log_g)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(r_g, st_g, cs_g, log_g)
    for _ in range(2):                      # a replay starts from the same initial state
        st_g.copy_(st0)
        cs_g.copy_(cs0)
        for n_log, o_log in log_g:
            n_log.fill_(-9)
            o_log.fill_(-9)
        graph.replay()
        torch.cuda.synchronize()
        for (n_e, o_e), (n_g, o_g) in zip(log_e, log_g):
            assert torch.equal(n_e, n_g)
            assert torch.equal(o_e, o_g)
        assert torch.equal(st_e, st_g)
        assert torch.equal(cs_e, cs_g)
    r_g.check_status()
    assert (torch.stack([n for n, _ in log_e]) > 0).any()   # some round committed a step
