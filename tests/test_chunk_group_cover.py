"""Host-side check of how the chunkwise backward's gradient kernel shares its units among CTAs.

Units are (batch row, chunk, value head), value head fastest; the Hv/Hk consecutive units of a
(batch row, chunk, kv head) form a group whose dq, dk are the sum over its value heads. CTAs
take whole groups from a counter: the i-th index handed out is group
((b NC + c) Hk + hk) with c = NC - 1 - i / (B Hk), b = (i mod B Hk) / Hk, hk = i mod Hk (last
chunk first: the reverse sweep's order), and a CTA runs its group's units in ascending value
head. Every group is then summed by one CTA in ascending head order, whichever CTA takes it:
the sum's association depends neither on the grid (the SM count), nor on the batch size, nor
on the order the CTAs reach the counter. The kernel runs alongside the reverse sweep only
where the sweep is one wave (B Hv Dv/64 CTAs at most the SM count) and there are more groups
than SMs. This mirrors the kernel's and the launcher's index arithmetic and checks the cover."""
import itertools
import random

import pytest


def group_of(i, B, NC, Hk):
    """The kernel's group for the i-th index taken."""
    per_c = B * Hk
    c, r = NC - 1 - i // per_c, i % per_c
    return ((r // Hk) * NC + c) * Hk + r % Hk


def overlaps(B, Hv, Hk, NC, nsplit, sms):
    """The launcher's choice: the gradient kernel alongside the reverse sweep."""
    return B * Hv * nsplit <= sms and NC * Hk * B > sms


def schedule(B, NC, Hk, rep, ctas, seed):
    """A run of the counter scheme: CTAs reach the counter in a random interleaving; each takes
    its first group at its start and the next one at the first unit of each group. Returns
    {cta: [unit, ...]} in the order each CTA runs them."""
    groups = B * NC * Hk
    rng = random.Random(seed)
    counter = 0
    pending = {}
    runs = {k: [] for k in range(ctas)}
    for k in rng.sample(range(ctas), ctas):              # first groups, in the order CTAs start
        pending[k] = counter
        counter += 1
    live = [k for k in range(ctas) if pending[k] < groups]
    while live:
        k = rng.choice(live)
        i = pending[k]
        g = group_of(i, B, NC, Hk)
        nxt = counter                                    # taken at the group's first unit
        counter += 1
        runs[k].extend(g * rep + hh for hh in range(rep))
        pending[k] = nxt
        if nxt >= groups:
            live.remove(k)
    return runs


@pytest.mark.parametrize("B,NC,Hk", [(1, 32, 16), (1, 4, 16), (8, 64, 16), (3, 5, 2), (1, 1, 1), (2, 7, 3)])
def test_group_order_is_a_bijection_last_chunk_first(B, NC, Hk):
    groups = B * NC * Hk
    gs = [group_of(i, B, NC, Hk) for i in range(groups)]
    assert sorted(gs) == list(range(groups))
    chunks = [(g // Hk) % NC for g in gs]
    assert chunks == sorted(chunks, reverse=True)        # the reverse sweep's order


@pytest.mark.parametrize("B,NC,Hk,rep,ctas", [
    (1, 32, 16, 4, 152),     # linattn-T2048 on a GB300
    (1, 4, 16, 4, 64),       # linattn-T256: fewer groups than SMs (grid = groups)
    (8, 64, 16, 2, 152),     # batched
] + [(B, NC, Hk, rep, ctas) for B, NC, Hk, rep, ctas in itertools.product((1, 3), (1, 2, 5), (1, 4), (1, 2, 4), (1, 2, 7))])
def test_every_unit_once_and_no_group_split(B, NC, Hk, rep, ctas):
    groups = B * NC * Hk
    ctas = min(ctas, groups)
    for seed in range(3):
        runs = schedule(B, NC, Hk, rep, ctas, seed)
        seen = sorted(u for us in runs.values() for u in us)
        assert seen == list(range(groups * rep))         # each unit once
        owner = {}
        for k, us in runs.items():
            for j in range(0, len(us), rep):
                block = us[j:j + rep]
                g = block[0] // rep
                assert block == [g * rep + hh for hh in range(rep)]   # a whole group, ascending heads
                assert owner.setdefault(g, k) == k


def test_batch_rows_map_to_the_same_group_sums():
    """Batch row b's group (c, hk) is group (b NC + c) Hk + hk; whichever CTA takes it, its
    units are the same value heads in the same order, so a B = 8 problem sums each group as
    eight B = 1 problems do."""
    NC, Hk, rep = 5, 3, 4
    for B in (1, 3, 8):
        for i in range(B * NC * Hk):
            g = group_of(i, B, NC, Hk)
            b, c, hk = g // Hk // NC, (g // Hk) % NC, g % Hk
            assert g == (b * NC + c) * Hk + hk
            assert [g * rep + hh for hh in range(rep)] == [((b * NC + c) * Hk + hk) * rep + hh for hh in range(rep)]


@pytest.mark.parametrize("name,B,Hv,Hk,NC,nsplit,expect", [
    ("linattn-T256", 1, 64, 16, 4, 2, False),
    ("linattn-T512", 1, 64, 16, 8, 2, False),
    ("linattn-T1024", 1, 64, 16, 16, 2, True),
    ("linattn-T2048", 1, 64, 16, 32, 2, True),
    ("batched", 8, 32, 16, 64, 2, False),                # the reverse sweep takes several waves
    ("long", 1, 64, 16, 512, 2, True),
    ("long-tp8", 1, 8, 2, 512, 2, True),
])
def test_which_shapes_overlap(name, B, Hv, Hk, NC, nsplit, expect):
    assert overlaps(B, Hv, Hk, NC, nsplit, 152) == expect, name
