"""The w2 GEMM's A-slot schedule, replayed on the host.

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
