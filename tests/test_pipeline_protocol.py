"""A discrete-event model of the GEMM kernel's per-stage barrier protocol (CPU
only), run under many random interleavings for the ring configurations the
planner produces.

Roles, as in qmoe_gemm_kernel: two TMA producer threads (even / odd stages),
two dequant sets (even / odd stages), NI MMA issuers (stage g to issuer
g mod NI).  Rings: NW weight slots, NB TMEM A slots, NB2 token-tile slots (a
multiple of NB) each with a "done" barrier that the stage's MMA commit
completes.  mbarriers are modelled phase-exactly with the hardware's parity
test (a wait on parity P passes while the barrier's current phase parity is not
P), so a waiter two phases behind would pass wrongly; the model flags that.

Checked: no deadlock; a weight slot is refilled only after the dequant set read
it; an A slot is rewritten only after the MMAs that read it completed; a token-
tile slot is refilled only after the MMAs that read it completed; every MMA
reads the A tile and the token tile of its own stage.
"""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.tx = 0
        self.phase = 0  # completed phases

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self, n=1, tx=0):
        self.pending -= n
        self.tx += tx
        assert self.pending >= 0
        self._maybe_complete()

    def complete_tx(self, n):
        self.tx -= n
        assert self.tx >= 0
        self._maybe_complete()

    def test(self, target):
        """Wait for the completion of phase `target` (0-based); target -1 is the
        phase before the first, which a fresh barrier reports complete."""
        ok = (self.phase & 1) != (target & 1)
        if ok:
            # the parity answer is right only while the barrier is at most one phase ahead
            assert self.phase <= target + 1, f"waiter two phases behind ({self.phase} vs {target})"
        return ok


def simulate(n_stages, NW, NB, NB2, NI, seed, DS=2):
    """DS dequant sets take stages g = s, s + DS, ... (each set's warps arrive as one)."""
    rng = random.Random(seed)
    wfull = [Bar(1) for _ in range(NW)]
    wempty = [Bar(16 // DS) for _ in range(NW)]
    afull = [Bar(16 // DS) for _ in range(NB)]
    done = [Bar(1) for _ in range(NB2)]
    wslot = [None] * NW        # stage whose weights the slot holds
    wread = [None] * NW        # last stage whose weights were read from the slot
    aslot = [None] * NB
    bslot = [None] * NB2
    mma_done = set()
    inflight = []              # async events: (kind, stage)

    def producer(p):
        for g in range(p, n_stages, 2):
            w, b = g % NW, g % NB2
            while not wempty[w].test(g // NW - 1):
                yield
            assert g < NW or wread[w] == g - NW, "weight slot refilled before it was read"
            wfull[w].arrive(1, tx=2)
            inflight.append(("w", g))
            while not done[b].test(g // NB2 - 1):
                yield
            assert g < NB2 or (g - NB2) in mma_done, "token-tile slot refilled before its MMAs completed"
            inflight.append(("b", g))
            yield

    def dequant(s):
        for g in range(s, n_stages, DS):
            w, a = g % NW, g % NB
            while not wfull[w].test(g // NW):
                yield
            assert wslot[w] == g and bslot[g % NB2] == g
            wread[w] = g
            wempty[w].arrive(16 // DS)
            yield  # conversion
            if NB2 != NB:
                gp = g - NB
                while not done[gp % NB2].test(gp // NB2 if gp >= 0 else -1):
                    yield
            assert g < NB or (g - NB) in mma_done, "A slot rewritten before its MMAs completed"
            aslot[a] = g
            afull[a].arrive(16 // DS)
            yield

    def issuer(i):
        for g in range(i, n_stages, NI):
            a = g % NB
            while not afull[a].test(g // NB):
                yield
            inflight.append(("mma", g))
            yield

    agents = [producer(0), producer(1)] + [dequant(s) for s in range(DS)] + [issuer(i) for i in range(NI)]
    live = list(agents)
    mma_queue = []
    steps = 0
    while live or inflight:
        steps += 1
        assert steps < 200000, "no progress (deadlock)"
        choices = [("agent", a) for a in live] + [("ev", k) for k in range(len(inflight))]
        kind, x = rng.choice(choices)
        if kind == "agent":
            try:
                next(x)
            except StopIteration:
                live.remove(x)
            continue
        ev, g = inflight.pop(x)
        if ev == "w":
            wslot[g % NW] = g
            wfull[g % NW].complete_tx(1)
        elif ev == "b":
            bslot[g % NB2] = g
            wfull[g % NW].complete_tx(1)
        else:
            # MMAs of one CTA execute in issue order; each reads its stage's A and token tiles
            mma_queue.append(g)
            g0 = mma_queue.pop(0)
            assert aslot[g0 % NB] == g0 and bslot[g0 % NB2] == g0, "MMA read another stage's operands"
            mma_done.add(g0)
            done[g0 % NB2].arrive(1)
    assert len(mma_done) == n_stages


CONFIGS = [
    # (NW, NB, NB2, NI): decode tiles (3 issuers, 6 A slots), mid (2 issuers, 4 slots), prefill (1 issuer)
    (16, 6, 12, 3), (16, 6, 6, 3), (14, 6, 18, 3), (8, 6, 12, 3),
    (10, 4, 8, 2), (10, 4, 4, 2), (10, 4, 4, 1), (6, 4, 8, 1), (2, 2, 4, 1), (4, 2, 2, 2),
]


@pytest.mark.parametrize("NW,NB,NB2,NI", CONFIGS)
def test_protocol_random_interleavings(NW, NB, NB2, NI):
    for seed in range(12):
        simulate(3 * NB2 + 2 * NW + 7, NW, NB, NB2, NI, seed)


# four dequant sets of four full-row warps: weight ring and token-tile ring multiples of 4
CONFIGS4 = [(16, 6, 12, 3), (12, 6, 12, 3), (8, 6, 12, 3), (12, 4, 8, 2), (8, 4, 4, 2), (12, 4, 4, 1), (8, 4, 8, 1)]


@pytest.mark.parametrize("NW,NB,NB2,NI", CONFIGS4)
def test_protocol_four_dequant_sets(NW, NB, NB2, NI):
    for seed in range(12):
        simulate(3 * NB2 + 2 * NW + 9, NW, NB, NB2, NI, seed, DS=4)


def test_model_detects_a_missing_wait():
    """The model is sharp: without the dequant sets' wait for the A slot's
    previous MMAs (rings of different depth), some interleaving rewrites an A
    slot too early."""
    found = False
    for seed in range(200):
        try:
            _simulate_without_aslot_wait(40, 16, 6, 12, 3, seed)
        except AssertionError as e:
            assert "A slot rewritten" in str(e) or "another stage" in str(e)
            found = True
            break
    assert found


def _simulate_without_aslot_wait(n_stages, NW, NB, NB2, NI, seed):
    """simulate() with NB2 != NB but the dequant's done wait left out (planted fault)."""
    rng = random.Random(seed)
    wfull = [Bar(1) for _ in range(NW)]
    wempty = [Bar(8) for _ in range(NW)]
    afull = [Bar(8) for _ in range(NB)]
    done = [Bar(1) for _ in range(NB2)]
    wslot, aslot, bslot = [None] * NW, [None] * NB, [None] * NB2
    mma_done, inflight, mma_queue = set(), [], []

    def producer(p):
        for g in range(p, n_stages, 2):
            w, b = g % NW, g % NB2
            while not wempty[w].test(g // NW - 1):
                yield
            wfull[w].arrive(1, tx=2)
            inflight.append(("w", g))
            while not done[b].test(g // NB2 - 1):
                yield
            inflight.append(("b", g))
            yield

    def dequant(s):
        for g in range(s, n_stages, 2):
            w, a = g % NW, g % NB
            while not wfull[w].test(g // NW):
                yield
            wempty[w].arrive(8)
            yield
            assert g < NB or (g - NB) in mma_done, "A slot rewritten before its MMAs completed"
            aslot[a] = g
            afull[a].arrive(8)
            yield

    def issuer(i):
        for g in range(i, n_stages, NI):
            while not afull[g % NB].test(g // NB):
                yield
            inflight.append(("mma", g))
            yield

    live = [producer(0), producer(1), dequant(0), dequant(1)] + [issuer(i) for i in range(NI)]
    while live or inflight:
        choices = [("agent", a) for a in live] + [("ev", k) for k in range(len(inflight))]
        kind, x = rng.choice(choices)
        if kind == "agent":
            try:
                next(x)
            except StopIteration:
                live.remove(x)
            continue
        ev, g = inflight.pop(x)
        if ev == "w":
            wslot[g % NW] = g
            wfull[g % NW].complete_tx(1)
        elif ev == "b":
            bslot[g % NB2] = g
            wfull[g % NW].complete_tx(1)
        else:
            mma_queue.append(g)
            g0 = mma_queue.pop(0)
            assert aslot[g0 % NB] == g0 and bslot[g0 % NB2] == g0, "MMA read another stage's operands"
            mma_done.add(g0)
            done[g0 % NB2].arrive(1)
