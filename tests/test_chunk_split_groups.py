"""Host-side check of how the chunkwise backward's gradient kernel and its reduction kernel share
the sum of dq, dk over the value heads of a kv head.

The gradient kernel's CTAs take contiguous ranges of (batch row, chunk, value head) units,
value head fastest, so a group of Hv/Hk consecutive units (one kv head and chunk) either lies
in one CTA's range, and leaves from it summed, or is split between CTAs, each of which leaves
one fp32 partial under the first head of its part; chunk_reduce_kernel (one block per CTA
boundary, the first boundary inside a group handles it) adds the parts. This mirrors the
kernels' index arithmetic and checks the cover: every split group is reduced exactly once,
over exactly the parts that were written, and no whole group is touched."""
import itertools

import pytest


def ranges(units, ctas):
    return [(i * units // ctas, (i + 1) * units // ctas) for i in range(ctas)]


def written_parts(units, ctas, rep, Hv):
    """(group, head of the part's first unit) for each partial the gradient kernel leaves, and
    the set of groups it completes itself."""
    parts, whole_groups = set(), set()
    for u_begin, u_end in ranges(units, ctas):
        for u in range(u_begin, u_end):
            h = u % Hv
            hh = h % rep
            g0 = u - hh
            whole = g0 >= u_begin and g0 + rep <= u_end
            glast = hh == rep - 1 or u + 1 == u_end
            if not glast:
                continue
            g = u // rep
            if whole:
                whole_groups.add(g)
            else:
                hs = h - (u - max(g0, u_begin))
                parts.add((g, hs))
    return parts, whole_groups


def reduced_parts(units, ctas, rep, Hv):
    """(group, part head) pairs that chunk_reduce_kernel reads, and how often each group is
    reduced."""
    read, count = set(), {}
    for i in range(1, ctas):
        ub = i * units // ctas
        if ub % rep == 0:
            continue
        g = ub // rep
        if (i - 1) * units // ctas > g * rep:
            continue
        starts = []
        for k in range(i - 1, ctas):
            us = g * rep if k == i - 1 else k * units // ctas
            if us >= (g + 1) * rep:
                break
            starts.append(us % Hv)
        count[g] = count.get(g, 0) + 1
        read.update((g, s) for s in starts)
    return read, count


@pytest.mark.parametrize("units,ctas,rep,Hv", [
    (2048, 152, 4, 64),      # linattn-T2048 on a GB300: 13.47 units per CTA
    (256, 152, 4, 64),       # fewer units than two per CTA
    (24, 24, 2, 4),          # one unit per CTA: every group split
    (24, 24, 3, 6),
    (32768, 152, 4, 64),
    (18, 7, 3, 6),
    (40, 40, 1, 4),          # one value head per kv head: nothing to sum
    (64, 64, 64, 64),        # one kv head for 64 value heads, one unit per CTA: 64 parts
    (128, 100, 32, 64),
] + [(r * m * n, c, r, r * m) for n, c, r, m in itertools.product((3, 7, 25), (2, 5, 13), (2, 3, 4), (1, 2))])
def test_split_groups_are_reduced_exactly_once(units, ctas, rep, Hv):
    if units % Hv or ctas > units:
        pytest.skip("units are whole (chunk, value head) rows; at most one CTA per unit")
    parts, whole = written_parts(units, ctas, rep, Hv)
    read, count = reduced_parts(units, ctas, rep, Hv)
    split_groups = {g for g, _ in parts}
    assert read == parts                                  # every partial is read, nothing else
    assert set(count) == split_groups and all(n == 1 for n in count.values())
    assert not (split_groups & whole)
    assert split_groups | whole == set(range(units // rep))   # every group leaves once
    for g in split_groups:                                # parts start at distinct heads of the group
        heads = sorted(s for gg, s in parts if gg == g)
        assert heads[0] == (g * rep) % Hv and len(set(heads)) == len(heads) <= rep
