"""Model check of the shared-memory ring protocol of the streaming kernels
(k_sparse_decode, k_page_scores): per consumer warp, R stages; the producer
issues chunk i into stage i mod R once the stage's `empty` barrier has
completed phase floor(i / R) - 1 (for i >= R), the copy lands later and
completes `full`'s phase; the consumer waits on `full` with parity
floor(i / R) mod 2, reads, and arrives on `empty`.  An mbarrier parity wait
only compares the parity of the current phase, so a wait two phases early
would pass: the check below runs the protocol under random interleavings and
copy latencies and asserts that every read sees its own chunk and that the
run never deadlocks.  CPU only."""
import random

import pytest


class Barrier:
    """Count-1 mbarrier: `phase` counts completed phases; a parity-P wait
    passes once the current (incomplete) phase has a parity other than P."""

    def __init__(self):
        self.phase = 0

    def complete(self):
        self.phase += 1

    def passes(self, parity):
        return (self.phase & 1) != parity


def run(R, n_chunks, seed, early_producer=False):
    rng = random.Random(seed)
    full = [Barrier() for _ in range(R)]
    empty = [Barrier() for _ in range(R)]
    stage = [None] * R          # chunk id held by each stage once its copy landed
    in_flight = []              # (land time, stage, chunk)
    t, issued, consumed, reads = 0, 0, 0, []
    while consumed < n_chunks:
        t += 1
        # copies land after a random delay (complete_tx completes full's phase)
        for item in sorted(in_flight):
            if item[0] <= t:
                in_flight.remove(item)
                _, s, c = item
                stage[s] = c
                full[s].complete()
        choice = rng.random()
        if choice < 0.5 and issued < n_chunks:          # producer step
            i = issued
            s = i % R
            ok = i < R or (early_producer or empty[s].passes(((i // R) - 1) & 1))
            if ok:
                in_flight.append((t + rng.randint(1, 12), s, i))
                issued += 1
        elif consumed < issued or in_flight:              # consumer step
            i = consumed
            s = i % R
            if full[s].passes((i // R) & 1):
                reads.append((i, stage[s]))
                consumed += 1
                empty[s].complete()
        if t > 20000:
            raise RuntimeError("no progress")
    return reads


@pytest.mark.parametrize("R", [1, 2, 3, 6])
def test_every_read_sees_its_own_chunk(R):
    for seed in range(300):
        reads = run(R, 40, seed)
        assert [c for _, c in reads] == list(range(40)), (R, seed)


def test_the_check_catches_a_producer_that_skips_the_empty_wait():
    """Without the empty-barrier wait the producer overwrites stages the
    consumer has not read yet and the full barrier runs phases ahead of the
    consumer's parity: the model must report a wrong read or a hang."""
    caught = 0
    for seed in range(100):
        try:
            reads = run(2, 40, seed, early_producer=True)
            caught += any(i != c for i, c in reads)
        except RuntimeError:                        # the consumer's parity never comes round again
            caught += 1
    assert caught > 0
