"""Host-side model of the chunk kernels' store order: no shared-memory tile is rewritten while a
bulk or TMA store that reads it may still be reading.

Bulk and TMA stores are grouped per issuing thread (`cp.async.bulk.commit_group`); a thread's
`cp.async.bulk.wait_group.read N` returns once all but its N newest groups have read their
sources. Each kernel issues its stores from fixed threads; this mirrors, per kernel, which
thread commits which tiles and where it waits, and checks every rewrite of a tile (by any
thread, after the block barrier that follows the wait) against the groups still reading it.
The sequences are written by hand from the kernels' code (chunk_prep_kernel,
chunk_sweep_kernel, chunk_dsweep_kernel, chunk_grad_kernel) and must be kept in step with it;
each kernel has a control that drops one wait and must fail. In the sweeps the math warps'
rewrites follow the copy warp's waits through mbarrier hand-offs; the model places each
rewrite at the earliest point those hand-offs allow."""
import pytest


class Stores:
    """The bulk groups of the store-issuing threads: lists of tile sets, oldest first."""

    def __init__(self):
        self.groups = {}

    def commit(self, thread, tiles):
        self.groups.setdefault(thread, []).append(set(tiles))

    def wait_read(self, thread, but=0):
        g = self.groups.get(thread, [])
        self.groups[thread] = g[len(g) - but:] if but else []

    def write(self, tiles, what):
        busy = set().union(*[t for g in self.groups.values() for t in g]) if self.groups else set()
        assert not (busy & set(tiles)), f"{what} rewritten while a store still reads it"


def sweep(NC, drop=None, infer=False):
    """chunk_sweep_kernel: the copy warp's issuing lane stores every tile. Per chunk c it stores the
    bf16 state (sop) once the math warps have written it, the previous chunk's y and v - u (ysg,
    rsg), and the staged fp32 checkpoint (group W's buffer c % 2 and the extra box ckx c % 2);
    then it waits until all but that newest group have read their tiles and releases sop, ysg
    and rsg to the math warps (fS), which go on with the next chunk, while it waits for the rest
    and refills group W's buffer c % 2 with chunk c + 2's operands. The inference forward
    (`infer`) stores only y: its release waits for every group, as the newest is y's."""
    st = Stores()
    T = "copy"
    st.write({"sop"}, "state operand of chunk 0")
    for c in range(NC):
        if not infer:                                  # the inference forward saves no state
            st.commit(T, {"sop"})
        if c > 0:
            st.commit(T, {"ysg"} if infer else {"ysg", "rsg"})
        if not infer:
            st.write({f"W{c % 2}", f"ckx{c % 2}"}, f"staged checkpoint of chunk {c}")
            st.commit(T, {f"W{c % 2}", f"ckx{c % 2}"})
            if drop != "fS":
                st.wait_read(T, but=1)
        elif drop == "fS":
            st.wait_read(T, but=1)                     # the wait that is right only with a checkpoint store
        else:
            st.wait_read(T)
        if c + 1 < NC:
            st.write({"sop"}, f"state operand of chunk {c + 1}")
            st.write({"ysg", "rsg"}, f"y / v - u staging of chunk {c}")
        if drop != "W":
            st.wait_read(T)
        if c + 2 < NC:
            st.write({f"W{c % 2}"}, f"group W of chunk {c + 2}")
    st.write({"ysg", "rsg"}, f"y / v - u staging of chunk {NC - 1}")
    st.commit(T, {"ysg", "rsg"})


def dsweep(NC, drop=None):
    """chunk_dsweep_kernel: the copy warp's issuing lane stores every tile. Per chunk (in reverse
    order) it stores dS_L (the high tile of shl) once the math warps have written it and releases
    shl (fS) after that store has read it; then it stores the chunk's [dY; dU] buffer, Delta and
    dv (dls, dvs) and, after they have been read, releases dls and dvs (fO) and refills that
    [dY; dU] buffer with the dY of the chunk two ahead. The math warps write the next chunk's dS
    operands after fS and the carry, its Delta and dv tiles after fO."""
    st = Stores()
    T = "copy"
    st.write({"shl"}, f"dS operands of chunk {NC - 1}")
    for k in range(NC):
        c, buf = NC - 1 - k, k & 1
        st.commit(T, {"shl"})
        if drop != "fS":
            st.wait_read(T)
        st.write({f"ydu{buf}", "dls", "dvs"}, f"dU rows, Delta and dv of chunk {c}")
        st.commit(T, {f"ydu{buf}", "dls", "dvs"})
        if k + 1 < NC:
            st.write({"shl"}, f"dS operands of chunk {c - 1}")
        if drop != "fO":
            st.wait_read(T)
        if k + 2 < NC:
            st.write({f"ydu{buf}"}, f"dY of chunk {c - 2}")


def grad(groups, rep, drop=None):
    """chunk_grad_kernel: per unit the decay table is written to stg; with the group's last head,
    thread 32 stores dq from stg, waits for that store's read, then stores dk from stg; it waits
    again at the next unit's top before the table is rewritten."""
    st = Stores()
    for g in range(groups):
        for hh in range(rep):
            if drop != "top":
                st.wait_read(32)
            st.write({"stg"}, f"decay table of unit {g * rep + hh}")
            if hh == rep - 1:
                st.write({"stg"}, f"dq tile of group {g}")
                st.commit(32, {"stg"})
                if drop != "between":
                    st.wait_read(32)
                st.write({"stg"}, f"dk tile of group {g}")
                st.commit(32, {"stg"})


def prep(units, rep, drop=None):
    """chunk_prep_kernel: thread 32 stores [Q; K] from kc, qc at a group's first unit and T diag(beta)
    from tcu per unit; it waits before the inversion (tcu is rewritten after it; the wait also
    covers the [Q; K] stores of the same unit) and, when the next unit starts another group,
    again before K and Q are fetched into kc, qc."""
    st = Stores()
    for u in range(units):
        if u % rep == 0:
            st.commit(32, {"kc", "qc"})
        if drop != "tcu":
            st.wait_read(32)
        st.write({"tcu"}, f"T diag(beta) of unit {u}")
        st.commit(32, {"tcu"})
        if u + 1 < units and (u + 1) % rep == 0:
            if drop != "kq":
                st.wait_read(32)
            st.write({"kc", "qc"}, f"K and Q of unit {u + 1}")


@pytest.mark.parametrize("NC", [1, 2, 3, 8, 32])
def test_sweeps_never_rewrite_a_tile_in_flight(NC):
    sweep(NC)
    sweep(NC, infer=True)
    dsweep(NC)


@pytest.mark.parametrize("groups,rep", [(1, 1), (3, 4), (5, 2)])
def test_grad_and_prep_never_rewrite_a_tile_in_flight(groups, rep):
    grad(groups, rep)
    prep(groups * rep, rep)


@pytest.mark.parametrize("fn,arg,drop", [
    (sweep, 3, "fS"), (sweep, 3, "W"), (dsweep, 2, "fS"), (dsweep, 3, "fO"),
    (grad, (2, 2), "top"), (grad, (1, 2), "between"), (prep, (8, 4), "tcu"),
])
def test_controls_without_a_wait_fail(fn, arg, drop):
    with pytest.raises(AssertionError, match="rewritten while a store still reads it"):
        fn(*arg, drop=drop) if isinstance(arg, tuple) else fn(arg, drop=drop)


def test_inference_release_must_wait_for_every_store():
    """With no checkpoint store the newest group is y's: releasing the staging tiles after
    `wait_group.read 1` (the training forward's wait) would let y's staging be rewritten."""
    with pytest.raises(AssertionError, match="rewritten while a store still reads it"):
        sweep(3, drop="fS", infer=True)
