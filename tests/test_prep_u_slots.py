"""Host-side check of the forward prep kernel's U staging ring.

U (fp32, [Dv/32][64][32] per unit) leaves prep by TMA stores of 8 KB boxes staged in shared
memory. The staging slots reuse buffers that are dead once a unit's products are done: slots
0-3 lie over T, the inversion scratch and the T operands, slots 4-5 over A. Per unit the boxes
go out in passes of up to three (one bulk group per pass, box j in slot j mod 6); before a pass
that would reuse a slot, the storing thread waits until at most one group (the previous pass)
is still reading. The next unit writes A after waiting for every group to finish reading when
Dv > 128, and T after waiting for every group in any case.

This mirrors that order and checks that no slot is written while a store may still read it,
for every Dv the tensor-core forward takes and over several consecutive units."""
import pytest

SLOTS = 6
A_SLOTS = {4, 5}
T_SLOTS = {0, 1, 2, 3}


class Ring:
    def __init__(self):
        self.groups = []          # per committed group: set of slots it reads, or None when done

    def wait_read_but(self, n):
        live = [i for i, g in enumerate(self.groups) if g is not None]
        for i in live[: max(0, len(live) - n)]:
            self.groups[i] = None

    def reading(self):
        out = set()
        for g in self.groups:
            if g is not None:
                out |= g
        return out


def run_units(Dv, units, a_wait=True):
    ring = Ring()
    for _ in range(units):
        # unit start: A is written (after a full wait only when Dv > 128)
        if a_wait and Dv > 128:
            ring.wait_read_but(0)
        assert not (ring.reading() & A_SLOTS), "A written while a U store still reads it"
        # the inversion writes T and its operands after a full wait
        ring.wait_read_but(0)
        assert not (ring.reading() & T_SLOTS)
        # U passes
        nb = Dv // 32
        for pass_, c0 in enumerate(range(0, Dv, 96)):
            n = min(96, Dv - c0)
            if 3 * (pass_ + 1) > SLOTS:
                ring.wait_read_but(1)
            slots = {(c0 // 32 + j) % SLOTS for j in range(3) if 32 * j < n}
            assert max(c0 // 32 + j for j in range(3) if 32 * j < n) < nb
            assert not (ring.reading() & slots), f"Dv={Dv}: slot rewritten while its store reads it"
            ring.groups.append(slots)
        if Dv <= 128:
            used = set().union(*(g for g in ring.groups if g is not None)) if ring.groups else set()
            assert not (used & A_SLOTS), "Dv <= 128 must leave the A slots unused"


@pytest.mark.parametrize("Dv", [64, 128, 192, 256])
def test_u_staging_slots_are_never_overwritten_in_flight(Dv):
    run_units(Dv, units=5)


@pytest.mark.parametrize("Dv", [192, 256])
def test_missing_wait_before_a_is_caught(Dv):
    """Control: without the wait before A (Dv > 128 uses the A slots), the check fires."""
    with pytest.raises(AssertionError, match="A written"):
        run_units(Dv, units=2, a_wait=False)
