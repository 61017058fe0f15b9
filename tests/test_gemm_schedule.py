"""The GEMMs' load schedules, replayed on the host: w2's A slots, and the
A loads deferred past the dependency wait with early weight loads.

The w2 kernel keeps A in a ring of A_SLOTS shared-memory slots outside its
STAGES-deep B ring, and gives A no barrier of its own.  A fill (one 256-K stage
of one m-tile's A) completes on the barrier of the ring stage it is issued with,
and slot f % A_SLOTS is reused by fill f + A_SLOTS.  That is safe only if,
when the producer issues fill f + A_SLOTS, it has already waited for the MMAs of
every ring stage that reads fill f.  It waits for the MMAs of ring stage r -
STAGES before issuing ring stage r, and MMAs complete in order.  These tests
replay the kernel's sequence: tile i of a CTA, stage kt, paired tiles (two
column blocks of one m-tile, the second re-reading the first's A) or unpaired.
They check that invariant for every K depth the kernel pairs, and for unpaired
tiles of any depth."""
import pytest

A_SLOTS, STAGES = 5, 4  # as in the w2 plan of csrc/kernels_gemm.cu


def replay(KT: int, paired: bool, tiles: int):
    """Per fill: the ring stage it is issued with and the ring stages reading it."""
    issued, readers = {}, {}
    r = 0  # ring stage index, in issue order (one per (tile, kt))
    for i in range(tiles):
        for kt in range(KT):
            f = (i >> 1 if paired else i) * KT + kt  # the fill this stage reads
            if not paired or i % 2 == 0:
                issued[f] = r
            readers.setdefault(f, []).append(r)
            r += 1
    return issued, readers


@pytest.mark.parametrize("paired,KT", [(True, kt) for kt in range(1, A_SLOTS + 1)] +
                         [(False, kt) for kt in range(1, 13)])
def test_slot_reuse_waits_for_the_last_reader(paired, KT):
    issued, readers = replay(KT, paired, tiles=64)
    for f, r_issue in issued.items():
        g = f + A_SLOTS
        if g not in issued:
            continue
        waited_through = issued[g] - STAGES  # MMAs of ring stages <= this are done
        assert max(readers[f]) <= waited_through, (paired, KT, f, readers[f], issued[g])


@pytest.mark.parametrize("KT", range(1, A_SLOTS + 1))
def test_a_pairs_fills_take_distinct_slots(KT):
    for q in range(20):
        slots = [(q * KT + kt) % A_SLOTS for kt in range(KT)]
        assert len(set(slots)) == KT


def test_one_more_stage_than_slots_would_not_be_safe():
    """The check above can fail: with a pair six stages deep, fill f + 5 is
    issued before the second tile has read fill f, which is why the kernel
    pairs only up to A_SLOTS stages."""
    issued, readers = replay(A_SLOTS + 1, True, tiles=16)
    bad = [f for f in issued if f + A_SLOTS in issued and max(readers[f]) > issued[f + A_SLOTS] - STAGES]
    assert bad


def paired_choice(MT: int, NT: int, KT: int, G: int = 152) -> bool:
    """The kernel's rule: pair when the A stages fit the slots and two-tile
    units add at most 1/32 to the busiest CTA's tile count."""
    per_cta = -(-MT * NT // G)
    per_cta_paired = 2 * -(-(MT * (NT // 2)) // G)
    return KT <= A_SLOTS and NT % 2 == 0 and per_cta_paired * 32 <= per_cta * 33


def test_pairing_rule_on_the_workloads():
    NT, KT = 2816 // 128, -(-704 // 256)
    assert paired_choice(540, NT, KT)          # prefill-sized (about 540 m-tiles): 80 vs 79 tiles
    assert not paired_choice(48, NT, KT)       # decode, 8 tokens (48 experts): 8 vs 7
    assert not paired_choice(127, NT, KT)      # decode, 64 tokens: 20 vs 19
    assert paired_choice(109, NT, KT)          # decode, 32 tokens: 16 vs 16
    assert not paired_choice(540, NT, -(-1536 // 256))  # six A stages do not fit the slots


# ---------------------------------------------------------------- early weight loads
# With early weight loads (w13's wide tiles, w2's small-batch plan beside the
# self-routed w13) the producer issues the weight loads of its first ring
# stages before its dependency wait and defers their A loads.  It waits once
# STAGES loads are outstanding, or when its loads end, and then issues the A
# loads of stages 0 .. n-1 from a closed form: load s belongs to tile
# b + (s // KT) * G at K step s % KT.  These tests replay the producer's
# sequence and check that the closed form names the same m-tile and K step
# as the deferred load in that stage, and that no stage is refilled before
# its A load was issued.


def producer_deferred(KT, STAGES, n_i, b, G):
    """(stage, tile, kt) of every load issued before the wait, in order."""
    out, stage = [], 0
    for i in range(n_i):
        for kt in range(KT):
            if len(out) == STAGES:
                return out  # the wait and the A loads come before this stage is refilled
            out.append((stage, b + i * G, kt))
            stage = (stage + 1) % STAGES
    return out


def closed_form(n, KT, b, G):
    return [(s, b + (s // KT) * G, s % KT) for s in range(n)]


@pytest.mark.parametrize("STAGES", [4, 6, 7])
@pytest.mark.parametrize("KT", [1, 2, 3, 11, 12])
@pytest.mark.parametrize("n_i", [1, 2, 3, 7])
def test_early_a_loads_match_the_deferred_stages(STAGES, KT, n_i):
    for b, G in ((0, 152), (5, 152), (151, 152), (3, 8)):
        deferred = producer_deferred(KT, STAGES, n_i, b, G)
        assert len(deferred) == min(STAGES, KT * n_i)
        assert deferred == closed_form(len(deferred), KT, b, G)
        # stages 0 .. n-1, each once: no stage holds two deferred loads
        assert [s for s, _, _ in deferred] == list(range(len(deferred)))
