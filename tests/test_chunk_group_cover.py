"""Host-side check of how the chunkwise backward's gradient kernel shares its units among CTAs.

Units are (batch row, chunk, value head), value head fastest; the Hv/Hk consecutive units of a
(batch row, chunk, kv head) form a group whose dq, dk are the sum over its value heads. The
kernel gives each CTA a contiguous range of whole groups (group range [i G / n, (i + 1) G / n)
for CTA i of n), so that every group is summed by one CTA in ascending head order: the sum's
association then depends neither on the grid (the SM count) nor on the batch size. This
mirrors the kernel's index arithmetic and checks the cover."""
import itertools

import pytest


def unit_ranges(groups, ctas, rep):
    """The kernel's (u_begin, u_end) per CTA."""
    return [((i * groups // ctas) * rep, ((i + 1) * groups // ctas) * rep) for i in range(ctas)]


def grid_of(groups, sms):
    return min(groups, sms)


@pytest.mark.parametrize("groups,sms,rep", [
    (512, 152, 4),           # linattn-T2048 on a GB300
    (64, 152, 4),            # linattn-T256: fewer groups than SMs
    (8192, 152, 2),          # batched
    (8192, 152, 4),          # long
] + list(itertools.product((1, 3, 7, 25, 153), (1, 2, 5, 152), (1, 2, 3, 4, 64))))
def test_every_unit_once_and_no_group_split(groups, sms, rep):
    ctas = grid_of(groups, sms)
    rs = unit_ranges(groups, ctas, rep)
    seen = []
    for b, e in rs:
        assert b % rep == 0 and e % rep == 0 and e > b      # whole groups, never empty
        seen.extend(range(b, e))
    assert seen == list(range(groups * rep))               # contiguous, ascending, each unit once
    sizes = [(e - b) // rep for b, e in rs]
    assert max(sizes) - min(sizes) <= 1                    # balanced to one group


def test_batch_rows_map_to_the_same_group_sums():
    """Batch row b's group (c, hk) is group (b NC + c) Hk + hk; whichever CTA takes it, its
    units are the same value heads in the same order, so a B = 8 problem sums each group as
    eight B = 1 problems do."""
    NC, Hk, rep = 5, 3, 4
    for B, sms in ((1, 152), (8, 152), (8, 7), (3, 2)):
        groups = B * NC * Hk
        owners = {}
        for i, (b, e) in enumerate(unit_ranges(groups, grid_of(groups, sms), rep)):
            for u in range(b, e):
                owners.setdefault(u // rep, set()).add(i)
                assert (u % rep) == (u - (u // rep) * rep)
        assert all(len(s) == 1 for s in owners.values())
