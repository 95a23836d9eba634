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


class Ring:
    """The kernel's ring position: a role starts at its own index and steps by its
    stride with a single wrap (as the device code does)."""

    def __init__(self, idx, phase=0):
        self.idx, self.phase = idx, phase

    def step(self, r, n):
        self.idx += r
        if self.idx >= n:
            self.idx -= n
            self.phase ^= 1

    def at(self, g, n, what):
        """Check the position against stage g's slot (g mod n) and lap parity."""
        assert 0 <= self.idx < n, f"{what} ring position {self.idx} outside {n} slots"
        assert self.idx == g % n, f"{what} ring position {self.idx} is not stage {g}'s slot {g % n}"
        assert self.phase == (g // n) & 1, f"{what} ring phase of stage {g}"
        return self.idx


def simulate(n_stages, NW, NB, NB2, NI, seed, DS=2, pair=False):
    """DS dequant sets take stages g = s, s + DS, ... (each set's warps arrive as one).
    Slot indices come from the kernel's ring stepping, checked against g mod n.
    An issued stage's MMAs enter the CTA's tensor-core queue in issue order and
    execute from its head at random later times.

    pair: the CTA-pair form.  Two CTAs walk the same stages, each with its own
    producers, dequant sets, weight ring and token-tile ring; the A barriers
    live in CTA 0 and count both CTAs' sets; CTA 0's issuers issue MMAs that read
    both CTAs' A slots and token tiles, and each stage's commit arrives on the
    "done" barrier of both CTAs."""
    rng = random.Random(seed)
    C = 2 if pair else 1
    wfull = [[Bar(1) for _ in range(NW)] for _ in range(C)]
    wempty = [[Bar(16 // DS) for _ in range(NW)] for _ in range(C)]
    afull = [Bar(C * (16 // DS)) for _ in range(NB)]
    done = [[Bar(1) for _ in range(NB2)] for _ in range(C)]
    wslot = [[None] * NW for _ in range(C)]   # stage whose weights the slot holds
    wread = [[None] * NW for _ in range(C)]   # last stage whose weights were read from the slot
    aslot = [[None] * NB for _ in range(C)]
    bslot = [[None] * NB2 for _ in range(C)]
    mma_done = set()
    inflight = []              # async events: (kind, cta, stage)

    def producer(c, p):
        wr, br = Ring(p), Ring(p)
        for g in range(p, n_stages, 2):
            w, b = wr.at(g, NW, "producer weight"), br.at(g, NB2, "producer token-tile")
            wr.step(2, NW)
            br.step(2, NB2)
            while not wempty[c][w].test(g // NW - 1):
                yield
            assert g < NW or wread[c][w] == g - NW, "weight slot refilled before it was read"
            wfull[c][w].arrive(1, tx=2)
            inflight.append(("w", c, g))
            while not done[c][b].test(g // NB2 - 1):
                yield
            assert g < NB2 or (g - NB2) in mma_done, "token-tile slot refilled before its MMAs completed"
            inflight.append(("b", c, g))
            yield

    def dequant(c, s):
        wr, ar = Ring(s), Ring(s)
        dr = Ring(s - NB + NB2, 1)  # the done barrier of stage g - NB (lap -1 for the first NB stages)
        for g in range(s, n_stages, DS):
            w, a = wr.at(g, NW, "dequant weight"), ar.at(g, NB, "dequant A")
            if NB2 != NB:
                # waits on done[(g - NB) mod NB2] at the parity of lap (g - NB) // NB2 (-1 before the first)
                assert 0 <= dr.idx < NB2 and dr.idx == (g - NB) % NB2, f"dequant done ring position {dr.idx}"
                assert dr.phase == ((g - NB) // NB2) & 1, f"dequant done ring phase of stage {g}"
            wr.step(DS, NW)
            ar.step(DS, NB)
            dr.step(DS, NB2)
            while not wfull[c][w].test(g // NW):
                yield
            assert wslot[c][w] == g and bslot[c][g % NB2] == g
            wread[c][w] = g
            wempty[c][w].arrive(16 // DS)
            yield  # conversion
            if NB2 != NB:
                gp = g - NB
                while not done[c][gp % NB2].test(gp // NB2 if gp >= 0 else -1):
                    yield
            assert g < NB or (g - NB) in mma_done, "A slot rewritten before its MMAs completed"
            aslot[c][a] = g
            afull[a].arrive(16 // DS)
            yield

    def issuer(i):
        ar, br = Ring(i), Ring(i)
        for g in range(i, n_stages, NI):
            a = ar.at(g, NB, "issuer A")
            br.at(g, NB2, "issuer token-tile")
            ar.step(NI, NB)
            br.step(NI, NB2)
            while not afull[a].test(g // NB):
                yield
            mma_queue.append(g)
            inflight.append(("exec", 0, g))
            yield

    agents = [producer(c, p) for c in range(C) for p in (0, 1)] + [dequant(c, s) for c in range(C) for s in range(DS)]
    agents += [issuer(i) for i in range(NI)]
    live = list(agents)
    mma_queue = []
    steps = 0
    while live or inflight:
        steps += 1
        assert steps < 400000, "no progress (deadlock)"
        choices = [("agent", a) for a in live] + [("ev", k) for k in range(len(inflight))]
        kind, x = rng.choice(choices)
        if kind == "agent":
            try:
                next(x)
            except StopIteration:
                live.remove(x)
            continue
        ev, c, g = inflight.pop(x)
        if ev == "w":
            wslot[c][g % NW] = g
            wfull[c][g % NW].complete_tx(1)
        elif ev == "b":
            bslot[c][g % NB2] = g
            wfull[c][g % NW].complete_tx(1)
        else:
            # MMAs execute in issue order; each reads its stage's A and token tiles (in both CTAs of a pair)
            g0 = mma_queue.pop(0)
            for cc in range(C):
                assert aslot[cc][g0 % NB] == g0 and bslot[cc][g0 % NB2] == g0, "MMA read another stage's operands"
            mma_done.add(g0)
            for cc in range(C):
                done[cc][g0 % NB2].arrive(1)
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


@pytest.mark.parametrize("NW,NB,NB2,NI,DS", [(8, 4, 4, 1, 4), (12, 4, 8, 1, 4), (8, 4, 4, 2, 4), (10, 4, 4, 1, 2),
                                            (16, 6, 12, 2, 4), (4, 4, 4, 1, 4)])
def test_protocol_cta_pairs(NW, NB, NB2, NI, DS):
    """The CTA-pair form: both CTAs' dequant sets arrive on CTA 0's A barriers,
    and every MMA reads both CTAs' operands of its own stage."""
    for seed in range(10):
        simulate(3 * NB2 + 2 * NW + 9, NW, NB, NB2, NI, seed, DS=DS, pair=True)


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
        wr, br = Ring(p), Ring(p)
        for g in range(p, n_stages, 2):
            w, b = wr.at(g, NW, "producer weight"), br.at(g, NB2, "producer token-tile")
            wr.step(2, NW)
            br.step(2, NB2)
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


def _planner_shapes():
    """(NW, NB, NB2, NI, DS) of every plan the planner makes for the Mixtral-8x7B
    int4 / int8 and DeepSeek-like shapes, automatic and with token tiles 16..256."""
    import weight_only_quantized_moe_gb300 as q
    from weight_only_quantized_moe_gb300 import _native as N
    from tests.test_abi import _layer_struct
    shapes = set()
    for kw in (dict(E=8, H=4096, I=14336, group_size=128, qt=N.QMOE_INT4_GROUP),
               dict(E=8, H=4096, I=14336, group_size=-1, qt=N.QMOE_INT8_PER_COL),
               dict(E=8, H=6144, I=16384, group_size=128, qt=N.QMOE_INT4_GROUP)):
        for M in (1, 16, 64, 256, 2048):
            for T in [0] + list(range(16, 257, 16)):
                for ring in (0, 1):
                    for pair in (0, 1):
                        try:
                            opts = q.make_options(token_tile=T, token_ring=ring, cta_pair=pair)
                            p = q.qmoe_describe_plan(_layer_struct(**kw), M, 2, opts, 152)
                        except Exception:
                            continue
                        shapes.add((p["w_stages"], p["ab_stages"], p["b_stages"], p["issuers"], p["dq_sets"],
                                    p["cta_pair"]))
    return sorted(shapes)


def test_protocol_every_planner_shape():
    """Every ring shape the planner produces (token tiles up to 256 rows, both
    token-tile ring depths, single CTAs and CTA pairs) passes the model, ring
    stepping included."""
    shapes = _planner_shapes()
    assert len(shapes) >= 8 and any(s[-1] for s in shapes)
    for NW, NB, NB2, NI, DS, pair in shapes:
        for seed in range(4):
            simulate(3 * NB2 + 2 * NW + 9, NW, NB, NB2, NI, seed, DS=DS, pair=bool(pair))


def test_model_detects_a_ring_smaller_than_the_set_count():
    """Two A slots with four dequant sets: sets 2 and 3 would start past the ring."""
    with pytest.raises(AssertionError, match="outside"):
        simulate(40, 8, 2, 4, 1, 0, DS=4)


def test_model_detects_an_a_ring_not_a_multiple_of_the_issuers():
    """Why the A ring is a multiple of the issuer count: with 4 slots and 3
    issuers, an issuer can reach stage g while the slot's barrier is still two
    phases behind (stage g - 4 belongs to another issuer), and the parity test
    passes wrongly; some interleaving shows it."""
    found = False
    for seed in range(60):
        try:
            simulate(60, 8, 4, 8, 3, seed, DS=4)
        except AssertionError as e:
            assert "another stage" in str(e) or "two phases" in str(e)
            found = True
            break
    assert found
