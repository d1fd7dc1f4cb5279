"""A model of the expert GEMM's barrier protocol, checked on the CPU.

The persistent tcgen05 GEMM (csrc/gemm_tc.cu) runs five kinds of actors over mbarriers whose
waits test only the parity of a phase: the weight producer (raw units, a ring of RAWS), the
activation producer (B stages in shared memory, a ring of three), four dequant groups that take
the 64-k sub-tiles round-robin and write them into the A stages in tensor memory (a ring of two
pipeline stages of two sub-tiles each), the MMA issuer, whose commits complete in issue order,
and the epilogue. In a cluster of two CTAs each activation producer's copy lands in both CTAs,
and each MMA commit releases the activation stage in both. A wait for phase k is sound only while
the barrier is at phase k or k + 1: if it is still at phase k - 1, that phase has the other
parity and the wait returns at once, before phase k has even begun. An arrival (or copy) meant
for phase k that lands while an earlier phase is still open is counted in that earlier phase.

`simulate` replays the committed protocol under random interleavings and random completion delays
and asserts, for every wait, that its barrier had reached the phase it waits for (no parity
aliasing) and, for every arrival and copy, that it lands in the phase it belongs to. The constants
are the kernel's two geometries (two A stages with three B stages and two sub-tiles per stage, or
two A and two B stages with four sub-tiles per stage), raw rings of four units (Q2_K units hold
four sub-tiles, Q8_0 units two), clusters of one, two and four CTAs.
`simulate_single_ring` replays the earlier one-ring protocol; with it the last tests show that the
model does catch a dequant group that skips its release wait, and the split-ring variant that
faulted on the GPU (six A stages over three B stages, dequant groups waiting for the B tile).
"""
import random

import pytest


class Violation(AssertionError):
    pass


class Bar:
    """An mbarrier: `expected` arrivals per phase, plus transaction bytes that must land too."""

    def __init__(self, name, expected):
        self.name, self.expected = name, expected
        self.phase = 0          # index of the phase in progress (= completed phases)
        self.arrived = 0
        self.tx_pending = 0

    def arrive(self, k, tx=0):
        if self.phase != k:
            raise Violation(f"{self.name}: arrival for phase {k} while phase {self.phase} is open")
        self.arrived += 1
        self.tx_pending += tx
        self._maybe_complete()

    def land(self, k):
        if self.phase != k:
            raise Violation(f"{self.name}: bytes for phase {k} landed in phase {self.phase}")
        self.tx_pending -= 1
        self._maybe_complete()

    def _maybe_complete(self):
        if self.arrived == self.expected and self.tx_pending == 0:
            self.phase += 1
            self.arrived = 0

    def done(self, k):
        """A wait for phase k (k < 0: the slot's first use, nothing to wait for)."""
        return k < 0 or self.phase > k

    def check_wait(self, k):
        # the kernel polls the parity of phase k: that is sound only while the barrier is at phase
        # k (in progress) or k + 1 (just completed); two phases off, the parity answers wrongly
        if k >= 0 and not (k <= self.phase <= k + 1):
            raise Violation(f"{self.name}: wait for phase {k} began at phase {self.phase} (parity alias)")


def simulate_single_ring(ng, stages, raws, n_items, stages_per_item, seed, skip_empty_wait=False, b_stages=None):
    """b_stages=None: the committed protocol (one full/empty pair per stage for A and B).
    b_stages=n: the variant with separate A (`stages`) and B (`n`) rings, in which the first
    dequant warp of a group waits for the stage's B tile before handing the stage to the MMA."""
    rng = random.Random(seed)
    kpu = ng  # stages per raw unit: each group takes exactly one stage of every unit
    n_stages = n_items * stages_per_item
    n_units = n_stages // kpu
    split = b_stages is not None
    full = [Bar(f"full[{i}]", 1 if split else 2) for i in range(stages)]  # group (+ producer, + bytes)
    empty = [Bar(f"empty[{i}]", 1) for i in range(stages)]     # MMA commit
    bfull = [Bar(f"b_full[{i}]", 1) for i in range(b_stages)] if split else full
    bempty = [Bar(f"b_empty[{i}]", 1) for i in range(b_stages)] if split else empty
    nb = b_stages if split else stages
    raw_full = [Bar(f"raw_full[{i}]", 1) for i in range(raws)]  # weight producer (+ bytes)
    raw_empty = [Bar(f"raw_empty[{i}]", ng) for i in range(raws)]  # one arrival per group
    acc_full = [Bar(f"acc_full[{i}]", 1) for i in range(2)]     # MMA commit after an item's last stage
    acc_empty = [Bar(f"acc_empty[{i}]", 1) for i in range(2)]   # the epilogue has read the accumulator
    pending = []  # (kind, target, phase) asynchronous completions: copies landing, MMAs finishing

    def weight_producer():
        for u in range(n_units):
            b = raw_empty[u % raws]
            k = u // raws - 1
            b.check_wait(k)
            while not b.done(k):
                yield
            raw_full[u % raws].arrive(u // raws, tx=1)
            pending.append(("land", raw_full[u % raws], u // raws))
            yield

    def act_producer():
        for g in range(n_stages):
            b = bempty[g % nb]
            k = g // nb - 1
            b.check_wait(k)
            while not b.done(k):
                yield
            bfull[g % nb].arrive(g // nb, tx=1)
            pending.append(("land", bfull[g % nb], g // nb))
            yield

    def dequant(grp):
        for g in range(grp, n_stages, ng):
            u = g // kpu
            rb = raw_full[u % raws]
            rb.check_wait(u // raws)
            while not rb.done(u // raws):
                yield
            if not skip_empty_wait:
                eb = empty[g % stages]
                k = g // stages - 1
                eb.check_wait(k)
                while not eb.done(k):
                    yield
            for _ in range(rng.randint(0, 3)):  # dequantization takes a while
                yield
            if split:  # the fold: B of this stage must have landed before the hand-over
                bb = bfull[g % nb]
                bb.check_wait(g // nb)
                while not bb.done(g // nb):
                    yield
            full[g % stages].arrive(g // stages)
            raw_empty[u % raws].arrive(u // raws)
            yield

    mma_inflight = []

    def mma():
        g = 0
        for item in range(n_items):
            buf, k = item & 1, (item >> 1) - 1  # the epilogue has drained item - 2's buffer
            ab = acc_empty[buf]
            ab.check_wait(k)
            while not ab.done(k):
                yield
            for _ in range(stages_per_item):
                fb = full[g % stages]
                fb.check_wait(g // stages)
                while not fb.done(g // stages):
                    yield
                mma_inflight.append(("stage", g))  # commits arrive when every earlier MMA completes
                g += 1
                yield
            mma_inflight.append(("acc", item))
            yield

    def epilogue():
        for item in range(n_items):
            buf, k = item & 1, item >> 1
            ab = acc_full[buf]
            ab.check_wait(k)
            while not ab.done(k):
                yield
            for _ in range(rng.randint(0, 6)):  # reading TMEM, SwiGLU, stores
                yield
            acc_empty[buf].arrive(k)
            yield

    actors = [weight_producer(), act_producer(), mma(), epilogue()] + [dequant(j) for j in range(ng)]
    steps = 0
    while actors or pending or mma_inflight:
        steps += 1
        if steps > 200000:
            raise Violation("no progress (deadlock)")
        r = rng.random()
        if pending and r < 0.25:
            kind, bar, k = pending.pop(rng.randrange(len(pending)))
            bar.land(k)
            continue
        if mma_inflight and r < 0.45:
            kind, v = mma_inflight.pop(0)  # in order
            if kind == "acc":
                acc_full[v & 1].arrive(v >> 1)
                continue
            empty[v % stages].arrive(v // stages)
            if split:
                bempty[v % nb].arrive(v // nb)
            continue
        if actors:
            a = rng.choice(actors)
            try:
                next(a)
            except StopIteration:
                actors.remove(a)
    assert [b.phase for b in acc_empty] == [(n_items + 1 - i) // 2 for i in range(2)]
    return full, empty, raw_full, raw_empty


def simulate(kpu, raws, n_items, stages_per_item, seed, cs=1, a_stages=2, b_stages=3, sub=2, groups=4,
             release_count=None):
    """The committed protocol for a cluster of `cs` CTAs that run the same item sequence
    (release_count: arrivals that release an activation stage; the protocol's is cs)."""
    rng = random.Random(seed)
    n_stages = n_items * stages_per_item
    n_subs = n_stages * sub
    n_units = n_subs // kpu
    ctas = []
    for c in range(cs):
        ctas.append(dict(
            a_full=[Bar(f"{c}:a_full[{i}]", sub) for i in range(a_stages)],      # one arrival per sub-tile
            a_empty=[Bar(f"{c}:a_empty[{i}]", 1) for i in range(a_stages)],      # local MMA commit
            b_full=[Bar(f"{c}:b_full[{i}]", 1) for i in range(b_stages)],        # own producer (+ every copy)
            b_empty=[Bar(f"{c}:b_empty[{i}]", release_count or cs) for i in range(b_stages)],  # every CTA's commit
            raw_full=[Bar(f"{c}:raw_full[{i}]", 1) for i in range(raws)],
            raw_empty=[Bar(f"{c}:raw_empty[{i}]", kpu) for i in range(raws)],    # one arrival per sub-tile
            acc_full=[Bar(f"{c}:acc_full[{i}]", 1) for i in range(2)],
            acc_empty=[Bar(f"{c}:acc_empty[{i}]", 1) for i in range(2)],
            inflight=[]))
    pending = []  # (barrier, phase) copies still in flight

    def weight_producer(c):
        B = ctas[c]
        for u in range(n_units):
            k = u // raws - 1
            B["raw_empty"][u % raws].check_wait(k)
            while not B["raw_empty"][u % raws].done(k):
                yield
            B["raw_full"][u % raws].arrive(u // raws, tx=1)
            pending.append((B["raw_full"][u % raws], u // raws))
            yield

    def act_producer(c):
        B = ctas[c]
        for S in range(n_stages):
            bb, k = B["b_empty"][S % b_stages], S // b_stages - 1
            bb.check_wait(k)
            while not bb.done(k):
                yield
            B["b_full"][S % b_stages].arrive(S // b_stages, tx=cs)  # every CTA's share lands here
            for peer in ctas:  # this CTA's share, multicast to every CTA of the cluster
                pending.append((peer["b_full"][S % b_stages], S // b_stages))
            yield

    def dequant(c, grp):
        B = ctas[c]
        for gs in range(grp, n_subs, groups):
            u, S = gs // kpu, gs // sub
            rb = B["raw_full"][u % raws]
            rb.check_wait(u // raws)
            while not rb.done(u // raws):
                yield
            eb, k = B["a_empty"][S % a_stages], S // a_stages - 1
            eb.check_wait(k)
            while not eb.done(k):
                yield
            for _ in range(rng.randint(0, 3)):  # dequantization and the tensor-memory store
                yield
            B["a_full"][S % a_stages].arrive(S // a_stages)
            B["raw_empty"][u % raws].arrive(u // raws)
            yield

    def mma(c):
        B = ctas[c]
        S = 0
        for item in range(n_items):
            buf, k = item & 1, (item >> 1) - 1
            B["acc_empty"][buf].check_wait(k)
            while not B["acc_empty"][buf].done(k):
                yield
            for _ in range(stages_per_item):
                for bar, kk in ((B["b_full"][S % b_stages], S // b_stages), (B["a_full"][S % a_stages], S // a_stages)):
                    bar.check_wait(kk)
                    while not bar.done(kk):
                        yield
                B["inflight"].append(("stage", S))  # the commits arrive when every earlier MMA completes
                S += 1
                yield
            B["inflight"].append(("acc", item))
            yield

    def epilogue(c):
        B = ctas[c]
        for item in range(n_items):
            buf, k = item & 1, item >> 1
            B["acc_full"][buf].check_wait(k)
            while not B["acc_full"][buf].done(k):
                yield
            for _ in range(rng.randint(0, 6)):
                yield
            B["acc_empty"][buf].arrive(k)
            yield

    actors = []
    for c in range(cs):
        actors += [weight_producer(c), act_producer(c), mma(c), epilogue(c)] + [dequant(c, g) for g in range(groups)]
    steps = 0
    while actors or pending or any(B["inflight"] for B in ctas):
        steps += 1
        if steps > 400000:
            raise Violation("no progress (deadlock)")
        r = rng.random()
        if pending and r < 0.25:
            bar, k = pending.pop(rng.randrange(len(pending)))
            bar.land(k)
            continue
        busy = [B for B in ctas if B["inflight"]]
        if busy and r < 0.45:
            B = rng.choice(busy)
            kind, v = B["inflight"].pop(0)  # in order
            if kind == "acc":
                B["acc_full"][v & 1].arrive(v >> 1)
                continue
            B["a_empty"][v % a_stages].arrive(v // a_stages)
            for peer in ctas:  # the multicast commit releases the activation stage everywhere
                peer["b_empty"][v % b_stages].arrive(v // b_stages)
            continue
        if actors:
            a = rng.choice(actors)
            try:
                next(a)
            except StopIteration:
                actors.remove(a)
    for B in ctas:
        assert [b.phase for b in B["acc_empty"]] == [(n_items + 1 - i) // 2 for i in range(2)]
        assert sum(b.phase for b in B["a_full"]) == n_stages
        assert sum(b.phase for b in B["b_full"]) == n_stages
        assert sum(b.phase for b in B["b_empty"]) == n_stages
        assert sum(b.phase for b in B["raw_full"]) == n_units
    return ctas


@pytest.mark.parametrize("geom,sub,a_stages,b_stages", [("wide", 2, 2, 3), ("small", 4, 2, 2)])
@pytest.mark.parametrize("cs", [1, 2, 4])
@pytest.mark.parametrize("fmt,kpu", [("q2_k", 4), ("q8_0", 2)])
def test_committed_protocol_has_no_parity_alias(fmt, kpu, cs, geom, sub, a_stages, b_stages):
    # the kernel's two tile geometries: 192-token tiles with two sub-tiles per stage, three
    # activation stages; 128-token tiles with four sub-tiles per stage, two activation stages
    for seed in range(40):
        # four pipeline stages per item, three items
        simulate(kpu, raws=4, n_items=3, stages_per_item=4, seed=seed, cs=cs, a_stages=a_stages,
                 b_stages=b_stages, sub=sub)


def test_committed_protocol_with_short_items():
    # items of one pipeline stage (K = 128, the smallest): every ring wraps within an item
    for seed in range(60):
        simulate(2, raws=4, n_items=5, stages_per_item=1, seed=seed, cs=2)


def test_model_catches_a_stage_released_by_one_cta_of_a_pair():
    # if one commit released an activation stage in a cluster of two, a producer could multicast
    # the next use of the stage into the peer before the peer's MMA had read it: the model must see it
    caught = 0
    for seed in range(60):
        try:
            simulate(4, raws=4, n_items=3, stages_per_item=4, seed=seed, cs=2, release_count=1)
        except Violation:
            caught += 1
    assert caught > 0


def test_model_catches_a_group_that_skips_the_empty_wait():
    # without the wait on the stage's release a dequant group arms a barrier phase that is
    # still open: the model must see it
    caught = 0
    for seed in range(50):
        try:
            simulate_single_ring(4, 4, 4, n_items=3, stages_per_item=16, seed=seed, skip_empty_wait=True)
        except Violation:
            caught += 1
    assert caught > 0


def test_split_rings_are_sound_only_with_no_more_a_than_b_stages():
    # equal rings: sound
    for seed in range(100):
        simulate_single_ring(4, 4, 4, n_items=3, stages_per_item=16, seed=seed, b_stages=4)
    # six A stages over three B stages: the B wait of a group can start two phases behind
    caught = 0
    for seed in range(100):
        try:
            simulate_single_ring(4, 6, 4, n_items=3, stages_per_item=16, seed=seed, b_stages=3)
        except Violation:
            caught += 1
    assert caught > 0
