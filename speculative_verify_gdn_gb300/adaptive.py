"""Adaptive speculation switch over device-side acceptance counters.

colibrì (ch.08 §4.1, the adaptive off-switch): once enough drafts have been proposed, drafting is
turned off when fewer than one in ten was accepted (there, at least 24 proposed and
accepted · 10 < proposed), since a verified-but-rejected draft costs more than it saves.

`AcceptStats` keeps the counters on the device (`spec_stats_accumulate` after each accept call:
proposed and accepted totals and the histogram of accepted lengths, exact integers) and reads them
only when asked, so the round loop never synchronises for them. `AdaptiveSwitch` is the host-side
rule on a snapshot of those counters.
"""
from dataclasses import dataclass

import torch

from . import _lib


class AcceptStats:
    """Acceptance counters of one draft length N: [proposed, accepted, hist[0..N]] on the device."""

    def __init__(self, N, device="cuda"):
        self.N = int(N)
        self.counts = torch.zeros(self.N + 3, dtype=torch.int64, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def update(self, n_acc, stream=None):
        """Add one accept call's counts (n_acc [B] int32 on the device); asynchronous."""
        _lib.spec_stats_accumulate(n_acc, self.N, self.counts, status=self.status, stream=stream)

    def reset(self):
        self.counts.zero_()
        self.status.zero_()

    def snapshot(self):
        """Host copy of the counters (synchronises with the device)."""
        c = [int(x) for x in self.counts.cpu().tolist()]
        st = int(self.status.item())
        if st:
            names = [v for k, v in _lib.STATUS_BITS.items() if st & k]
            raise _lib.GdnError("spec_stats_accumulate: device status 0x%x (%s)" % (st, ", ".join(names)))
        return StatsSnapshot(proposed=c[0], accepted=c[1], hist=c[2:])


@dataclass(frozen=True)
class StatsSnapshot:
    proposed: int
    accepted: int
    hist: list

    @property
    def rate(self):
        return self.accepted / self.proposed if self.proposed else 0.0

    @property
    def mean_accepted(self):
        seqs = sum(self.hist)
        return self.accepted / seqs if seqs else 0.0


class AdaptiveSwitch:
    """Drafting stays on unless at least `min_proposed` drafts were proposed and the accepted share
    is below num / den (integer comparison accepted · den < proposed · num). The defaults are the
    rule quoted above: 24 proposals, one in ten."""

    def __init__(self, min_proposed=24, num=1, den=10):
        if min_proposed < 0 or num < 0 or den <= 0:
            raise ValueError("min_proposed >= 0, num >= 0 and den > 0 required")
        self.min_proposed, self.num, self.den = int(min_proposed), int(num), int(den)

    def enabled(self, snap: StatsSnapshot) -> bool:
        if snap.proposed < self.min_proposed:
            return True
        return snap.accepted * self.den >= snap.proposed * self.num

    def draft_count(self, snap: StatsSnapshot, N: int) -> int:
        """Drafts to propose in the next round: N while enabled, else 0."""
        return int(N) if self.enabled(snap) else 0
