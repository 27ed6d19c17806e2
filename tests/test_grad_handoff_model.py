"""Host-side model of the hand-off from the reverse sweep to the gradient kernel when the two run
side by side.

Each reverse-sweep CTA (one per block of 64 value rows of a head) goes through the chunks from
the last; its copy warp's issuing lane commits, per chunk handled k-th, a bulk group A_k (dS_L)
after the math warps' bH hand-off and a group B_k ([dY; dU], Delta, dv) after their bU
hand-off. The math warps write the chunk's f partials after their bR arrival and its dbeta
partials after their bU arrival, so the copy warp knows them written once it has waited for
their next arrival at bH (chunk k + 1), or after the CTA's final barrier. At every second chunk
(odd k > 1), once that chunk's fO release and fetches are done, the copy warp waits until at
most four of its bulk groups are pending (`cp.async.bulk.wait_group 4`: those groups' writes
complete) and adds 1 to the ready counters of the chunks handled three and two before; after
its loop (all groups complete) and the final barrier, to the chunks left. A gradient-kernel
group starts once the counters of its chunk reach nsplit for each of its value heads.

The sequence is written by hand from chunk_dsweep_kernel's copy-warp loop and must be kept in
step with it; the checks: a chunk is published only when all its stores are complete and its
partials written, each chunk exactly once per CTA, and controls (a shorter lag, a wait for
fewer groups) fail."""
import pytest


def dsweep_publish(NC, lag=2, keep=4, every=2):
    """The copy warp of one reverse-sweep CTA: the events in program order. Returns the list of
    (k_published, pending_groups_at_publish, partials_known) per publish."""
    pending = []                 # bulk groups not yet complete, oldest first: ("A"|"B", k)
    partials_known = -1          # highest k whose f and dbeta partials the copy warp knows written
    out = []

    def wait_group(n):
        del pending[:max(0, len(pending) - n)]

    for k in range(NC):
        # wait bH(k): the math warps have written chunk k's dS parts, and before that chunk
        # k - 1's partials
        partials_known = max(partials_known, k - 1)
        pending.append(("A", k))
        # wait bR(k); copy P; wait read; arrive fS
        # wait bU(k); copy T; the block's outputs
        pending.append(("B", k))
        # wait mS(k); copies; wait read; arrive fO; fetch
        if k > 1 and (k % every) == every - 1:
            wait_group(keep)
            for j in (k - lag - 1, k - lag):
                out.append((j, list(pending), partials_known))
    wait_group(0)                # bulk_wait_all after the loop
    partials_known = NC - 1      # the CTA's final barrier: every math-warp write precedes it
    published = {j for j, _, _ in out}
    for j in range(NC):                                  # chunk indices descending
        if j not in published:
            out.append((j, list(pending), partials_known))
    return out


def check(NC, **kw):
    pubs = dsweep_publish(NC, **kw)
    ks = [j for j, _, _ in pubs]
    assert sorted(ks) == list(range(NC)), "each chunk published once"
    for j, pending, known in pubs:
        assert not any(kk == j for _, kk in pending), f"chunk {j} published with its stores pending"
        assert known >= j, f"chunk {j} published before its partials are known written"
    return pubs


@pytest.mark.parametrize("NC", [1, 2, 3, 4, 5, 6, 7, 8, 31, 32, 33, 512])
def test_each_chunk_published_once_after_its_writes(NC):
    pubs = check(NC)
    # what the loop leaves is what the kernel publishes after its final barrier: chunk indices
    # (1 if NC - 1 is odd, else 2) down to 0, those below NC
    in_loop = sum(1 for k in range(NC) if k > 1 and k % 2 == 1) * 2
    start = 1 if (NC - 1) % 2 == 1 else 2
    after = [NC - 1 - cc for cc in range(start, -1, -1) if cc < NC]
    assert [j for j, _, _ in pubs[in_loop:]] == after


@pytest.mark.parametrize("NC", [1, 2, 5, 8, 32, 33])
def test_chunks_are_published_last_first(NC):
    """The gradient kernel takes groups last chunk first: the publication order matches."""
    chunks = [NC - 1 - j for j, _, _ in check(NC)]
    assert chunks == sorted(chunks, reverse=True)


@pytest.mark.parametrize("kw", [
    dict(lag=1, keep=4),         # the chunks handled two and one before: the latter's B group may be pending
    dict(lag=2, keep=5),         # a wait that leaves five groups pending: chunk k - 3's B group may be too
    dict(lag=0, keep=2),         # the chunk just handled: its partials are not known written
])
def test_controls_fail(kw):
    with pytest.raises(AssertionError):
        for NC in (4, 5, 8, 32):
            check(NC, **kw)
