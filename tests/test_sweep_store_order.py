"""Host-side check of the sweeps' store order (chunk_sweep_kernel, chunk_dsweep_kernel).

Per chunk the sweep's thread 0 commits two groups of bulk stores: the chunk-start state (the
bf16 operand `sop` and the fp32 checkpoint tile `ckst`), and, while the chunk's first product
runs, the previous chunk's y and v - u (staging tiles `ysg`, `rsg`). Its waits: at the top of a
chunk, all groups but the newest have read their tiles (all of them for the first two chunks);
before the state stores, all groups; before the epilogue after the last chunk, all groups.

This mirrors that order and checks that no staging tile is rewritten while a committed store may
still read it, for one chunk and several; a control drops the wait before the last epilogue."""
import pytest

from test_prep_u_slots import Ring


def run_sweep(NC, final_wait=True):
    ring = Ring()

    def write(tiles, what):
        assert not (ring.reading() & tiles), f"{what} rewritten while a store still reads it"

    def epilogue(cc):
        write({"ysg", "rsg"}, f"y / v - u staging of chunk {cc}")
        ring.groups.append({"ysg", "rsg"})

    for c in range(NC):
        ring.wait_read_but(1 if c >= 2 else 0)
        write({"sop", "ckst"}, f"state staging of chunk {c}")
        ring.wait_read_but(0)
        ring.groups.append({"sop", "ckst"})
        if c > 0:
            epilogue(c - 1)
    if final_wait:
        ring.wait_read_but(0)
    epilogue(NC - 1)


@pytest.mark.parametrize("NC", [1, 2, 3, 8, 32])
def test_staging_tiles_are_never_rewritten_in_flight(NC):
    run_sweep(NC)


@pytest.mark.parametrize("NC", [2, 5])
def test_missing_wait_before_the_last_epilogue_is_caught(NC):
    with pytest.raises(AssertionError, match="staging of chunk"):
        run_sweep(NC, final_wait=False)


def test_one_chunk_needs_no_final_wait():
    run_sweep(1, final_wait=False)


def run_dsweep(NC, wait_each_chunk=True):
    """chunk_dsweep_kernel, chunks in reverse: [dY; dU] double-buffered (dY of the next chunk is
    loaded into the other buffer), one group per chunk storing [dY; dU], Delta and dv from their
    tiles. Thread 0 waits for all groups once per chunk, before that load and the tile writes."""
    ring = Ring()

    def write(tiles, what):
        assert not (ring.reading() & tiles), f"{what} rewritten while a store still reads it"

    write({"ydu0"}, "dY buffer 0")
    for k in range(NC):
        buf = k & 1
        if wait_each_chunk:
            ring.wait_read_but(0)
        if k + 1 < NC:
            write({f"ydu{buf ^ 1}"}, f"dY buffer {buf ^ 1}")
        write({"dls", "dvs", f"ydu{buf}"}, f"Delta, dv and dU tiles of chunk {k}")
        ring.groups.append({f"ydu{buf}", "dls", "dvs"})


@pytest.mark.parametrize("NC", [1, 2, 3, 32])
def test_reverse_sweep_tiles_are_never_rewritten_in_flight(NC):
    run_dsweep(NC)


def test_reverse_sweep_without_its_wait_is_caught():
    with pytest.raises(AssertionError, match="rewritten while a store still reads it"):
        run_dsweep(3, wait_each_chunk=False)
