"""Adaptive speculation switch: the counting oracle and the off rule pinned to the page's
statement (colibrì ch.08 §4.1: off once at least 24 drafts were proposed and accepted · 10 <
proposed), the host policy checked against the oracle, and (GPU) the device counters
spec_stats_accumulate bit-exact against the oracle's counts."""
import numpy as np
import pytest
import torch

import oracle
from speculative_verify_gdn_gb300.adaptive import AcceptStats, AdaptiveSwitch, StatsSnapshot


def test_accept_stats_oracle_worked_example():
    # N = 5, two calls: n = [0, 2, 2, 5] then [5, 1]: 6 sequences x 5 proposals; 15 accepted
    proposed, accepted, hist, bad = oracle.accept_stats([[0, 2, 2, 5], [5, 1]], 5)
    assert proposed == 30 and accepted == 15 and not bad
    assert hist == [1, 1, 2, 0, 0, 2]
    # invariants that hold for any input: every sequence lands in one bin, accepted = Σ k hist[k]
    g = np.random.default_rng(0)
    calls = [g.integers(0, 9, size=13) for _ in range(4)]
    p2, a2, h2, b2 = oracle.accept_stats(calls, 8)
    assert sum(h2) == 52 and p2 == 52 * 8 and a2 == sum(k * h for k, h in enumerate(h2))
    assert a2 == int(sum(c.sum() for c in calls)) and not b2


def test_accept_stats_oracle_bad_count():
    proposed, accepted, hist, bad = oracle.accept_stats([[3, -1, 9]], 4)
    assert bad and proposed == 12 and accepted == 3 and hist == [0, 0, 0, 1, 0]


@pytest.mark.parametrize("proposed,accepted,on", [
    (24, 2, False),      # 20 < 24: off (the page's condition)
    (24, 3, True),       # 30 >= 24: on
    (23, 0, True),       # fewer than 24 proposed: the rule does not apply yet
    (240, 23, False), (240, 24, True), (0, 0, True)])
def test_off_rule_pinned_to_the_page(proposed, accepted, on):
    assert oracle.adaptive_enabled(proposed, accepted) == on
    assert AdaptiveSwitch().enabled(StatsSnapshot(proposed, accepted, [0])) == on


def test_switch_matches_oracle_on_a_grid():
    for mp, num, den in [(24, 1, 10), (0, 1, 4), (100, 3, 10)]:
        sw = AdaptiveSwitch(mp, num, den)
        for p in range(0, 130, 7):
            for a in range(0, p + 1, 3):
                assert sw.enabled(StatsSnapshot(p, a, [0])) == \
                    oracle.adaptive_enabled(p, a, mp, num, den), (mp, num, den, p, a)
                assert sw.draft_count(StatsSnapshot(p, a, [0]), 8) in (0, 8)


def test_snapshot_rates():
    s = StatsSnapshot(proposed=40, accepted=10, hist=[2, 1, 0, 1, 1])
    assert s.rate == 0.25 and s.mean_accepted == 2.0
    assert StatsSnapshot(0, 0, [0]).rate == 0.0


@pytest.mark.gpu
def test_device_counters_match_oracle(gdnlib):
    g = np.random.default_rng(5)
    N = 8
    st = AcceptStats(N)
    calls = []
    for B in (64, 1, 300):
        n = g.integers(0, N + 1, size=B).astype(np.int32)
        calls.append(n)
        st.update(torch.from_numpy(n).cuda())
    snap = st.snapshot()
    proposed, accepted, hist, bad = oracle.accept_stats(calls, N)
    assert not bad
    assert (snap.proposed, snap.accepted, snap.hist) == (proposed, accepted, hist)
    # a count outside [0, N] is reported and adds only its proposals
    st.reset()
    n = torch.tensor([1, 9, -2, 8], dtype=torch.int32, device="cuda")
    st.update(n)
    torch.cuda.synchronize()
    assert int(st.status.item()) & 0x1
    c = st.counts.cpu().tolist()
    assert c[0] == 4 * N and c[1] == 9 and c[2:] == [0, 1, 0, 0, 0, 0, 0, 0, 1]
    # N = 0 (nothing drafted): every sequence lands in bin 0
    st0 = AcceptStats(0)
    st0.update(torch.zeros(5, dtype=torch.int32, device="cuda"))
    s0 = st0.snapshot()
    assert (s0.proposed, s0.accepted, s0.hist) == (0, 0, [5])
