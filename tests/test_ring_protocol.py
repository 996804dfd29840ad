"""Model check of the shared-memory ring protocol of the streaming kernels
(k_sparse_decode in attention.cuh, k_page_scores in select.cuh), CPU only.

Per consumer warp there are R stages, each with a `full` and an `empty`
mbarrier of count one.  The producer lane issues chunk i into stage i mod R
once the stage's `empty` barrier passes its parity test (always for i < R),
the copy lands later and completes `full`'s phase; the consumer waits on
`full`, reads the stage and arrives on `empty`.  After an abort the producer
waits on `full` for its last R issued chunks, so that no copy is left in
flight.  An mbarrier parity wait only compares the parity of the current
phase, so a wait two phases early would pass; the check runs the protocol
under random interleavings and copy latencies.

The three parity expressions (producer, consumer, drain) and the stage
index are read from each kernel's source and evaluated here, so the check
covers the code as written: every read sees its own chunk, the run never
deadlocks, and the drain's waits all end.  Planted mistakes in the
expressions are caught.
"""
import os
import random
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCES = {"k_sparse_decode": "attention.cuh", "k_page_scores": "select.cuh"}


def _code(text):
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def _as_python(expr, counter, ring):
    """A C parity expression over (counter, ring) as a function of (i, R)
    (the operands are non-negative where it is evaluated, so C's integer
    division is Python's floor division)."""
    e = re.sub(r"\b%s\b" % re.escape(counter), "i", expr)
    e = re.sub(r"\b%s\b" % re.escape(ring), "R", e)
    e = e.replace("/", "//")
    assert re.fullmatch(r"[iR0-9 ()+\-*/&%]+", e), e
    return eval("lambda i, R: " + e)           # the expression is a few integer operators on i and R


class Protocol:
    def __init__(self, producer, consumer, drain, stage, text=None):
        self.producer, self.consumer, self.drain, self.stage = producer, consumer, drain, stage
        self.text = text or {}


def protocol_of(kernel):
    """The ring protocol of `kernel` as its source writes it."""
    code = _code(open(os.path.join(ROOT, "kv_cache_page_build_b300", "csrc", SOURCES[kernel])).read())
    m = re.search(r"if \((\w+) < (\w+) \|\| mbar_test_wait\(&empty\[s\], "
                  r"static_cast<uint32_t>\((.+?)\)\)\) \{", code)
    counter, ring, prod = m.groups()
    cons = re.search(r"mbar_wait\(&full\[s\], static_cast<uint32_t>\((.+?)\)(?:, \w+)?\)", code).group(1)
    dm = re.search(r"for \(int j = max\(0, (\w+) - (\w+)\); j < \1; \+\+j\) "
                   r"mbar_wait\(&full\[lane \* \2 \+ j % \2\], static_cast<uint32_t>\((.+?)\)(?:, \w+)?\)", code)
    assert dm and dm.group(1) == counter and dm.group(2) == ring
    drain = dm.group(3)
    st = re.search(r"const int s = lane \* %s \+ %s %% %s;" % (ring, counter, ring), code)
    assert st, "producer stage index"
    assert re.search(r"const int s = \w+ \* %s \+ %s %% %s;" % (ring, counter, ring),
                     code[code.index(cons) - 400:]), "consumer stage index"
    return Protocol(_as_python(prod, counter, ring), _as_python(cons, counter, ring),
                    _as_python(drain.replace("j", counter), counter, ring), lambda i, R: i % R,
                    dict(producer=prod, consumer=cons, drain=drain))


class Barrier:
    """Count-1 mbarrier: `phase` counts completed phases; a parity-P wait
    passes once the current (incomplete) phase has a parity other than P."""

    def __init__(self):
        self.phase = 0

    def complete(self):
        self.phase += 1

    def passes(self, parity):
        return (self.phase & 1) != parity


def run(proto, R, n_chunks, seed, abort_at=None):
    """One producer/consumer pair over n_chunks; returns (reads, drain_ok).
    abort_at: stop the consumer after that many reads, land every copy in
    flight and check that the producer's drain waits all pass."""
    rng = random.Random(seed)
    full = [Barrier() for _ in range(R)]
    empty = [Barrier() for _ in range(R)]
    stage = [None] * R          # chunk id held by each stage once its copy landed
    in_flight = []              # (land time, stage, chunk)
    t, issued, consumed, reads = 0, 0, 0, []
    target = n_chunks if abort_at is None else abort_at
    while consumed < target:
        t += 1
        for item in sorted(in_flight):            # copies land after a random delay
            if item[0] <= t:
                in_flight.remove(item)
                _, s, c = item
                stage[s] = c
                full[s].complete()
        if rng.random() < 0.5 and issued < n_chunks:        # producer step
            i = issued
            s = proto.stage(i, R)
            if i < R or empty[s].passes(proto.producer(i, R)):
                in_flight.append((t + rng.randint(1, 12), s, i))
                issued += 1
        elif consumed < issued:                             # consumer step
            i = consumed
            s = proto.stage(i, R)
            if full[s].passes(proto.consumer(i, R)):
                reads.append((i, stage[s]))
                consumed += 1
                empty[s].complete()
        if t > 20000:
            raise RuntimeError("no progress")
    for _, s, c in sorted(in_flight):                       # abort: every copy lands
        stage[s] = c
        full[s].complete()
    drain_ok = all(full[proto.stage(j, R)].passes(proto.drain(j, R)) for j in range(max(0, issued - R), issued))
    return reads, drain_ok


@pytest.mark.parametrize("kernel", sorted(SOURCES))
def test_protocol_is_read_from_the_source(kernel):
    p = protocol_of(kernel)
    assert set(p.text) == {"producer", "consumer", "drain"}
    # chunk i's copy completes full's phase i // R, and its stage was last
    # emptied in phase i // R - 1
    for R in (1, 2, 3, 6):
        for i in range(R, 5 * R):
            assert p.consumer(i, R) == (i // R) & 1 and p.producer(i, R) == (i // R - 1) & 1


@pytest.mark.parametrize("kernel", sorted(SOURCES))
def test_consumer_fast_path_tests_the_same_phase(kernel):
    """Where a consumer first tests its stage without waiting (a chunk that
    has landed is taken at once), the test uses the same parity as the
    modelled wait, so the model covers both paths."""
    code = _code(open(os.path.join(ROOT, "kv_cache_page_build_b300", "csrc", SOURCES[kernel])).read())
    fast = re.findall(r"mbar_try_wait\(&full\[s\], static_cast<uint32_t>\((.+?)\)\)", code)
    for expr in fast:
        assert expr == protocol_of(kernel).text["consumer"]
    if kernel == "k_sparse_decode":
        assert fast, "the attention's consumers test a landed chunk first"


@pytest.mark.parametrize("kernel", sorted(SOURCES))
@pytest.mark.parametrize("R", [1, 2, 3, 6])
def test_every_read_sees_its_own_chunk(kernel, R):
    p = protocol_of(kernel)
    for seed in range(200):
        reads, drain_ok = run(p, R, 40, seed)
        assert [c for _, c in reads] == list(range(40)), (kernel, R, seed)
        assert drain_ok


@pytest.mark.parametrize("kernel", sorted(SOURCES))
@pytest.mark.parametrize("R", [1, 2, 3])
def test_drain_after_an_abort_ends(kernel, R):
    p = protocol_of(kernel)
    for seed in range(200):
        reads, drain_ok = run(p, R, 40, seed, abort_at=seed % 37)
        assert [c for _, c in reads] == list(range(len(reads)))
        assert drain_ok, (kernel, R, seed)


def release_is_guarded(kernel):
    """Whether the consumer arrives on `empty` only for a stage whose wait
    succeeded (`if (lane == 0 && <flag>) mbar_arrive(&empty[s]);`)."""
    code = _code(open(os.path.join(ROOT, "kv_cache_page_build_b300", "csrc", SOURCES[kernel])).read())
    m = re.search(r"if \(lane == 0( && \w+)?\) mbar_arrive\(&empty\[s\]\);", code)
    assert m, "consumer release"
    return m.group(1) is not None


def run_abort(proto, R, n_chunks, seed, abort_at, guarded):
    """The abort as the kernels run it: after abort_at reads the consumer
    stops waiting but goes on over its remaining chunks, releasing a stage
    only when `guarded` is false; the producer notices the abort a random
    number of steps later.  Returns (a copy was issued into a stage whose
    previous copy was still in flight, the drain's waits all pass)."""
    rng = random.Random(seed)
    full = [Barrier() for _ in range(R)]
    empty = [Barrier() for _ in range(R)]
    in_flight = []
    t, issued, consumed, aborted, notice, overlap = 0, 0, 0, False, rng.randint(0, 8), False
    while True:
        t += 1
        for item in sorted(in_flight):
            if item[0] <= t:
                in_flight.remove(item)
                full[item[1]].complete()
        producing = issued < n_chunks and (not aborted or notice > 0)
        if rng.random() < 0.5 and producing:
            if aborted:
                notice -= 1
            i = issued
            s = proto.stage(i, R)
            if i < R or empty[s].passes(proto.producer(i, R)):
                overlap |= any(x[1] == s for x in in_flight)
                in_flight.append((t + rng.randint(1, 12), s, i))
                issued += 1
        elif not aborted:
            if consumed == abort_at:
                aborted = True
            elif consumed < issued and full[proto.stage(consumed, R)].passes(proto.consumer(consumed, R)):
                empty[proto.stage(consumed, R)].complete()
                consumed += 1
        elif consumed < n_chunks:                           # skipped without a wait
            if not guarded:
                empty[proto.stage(consumed, R)].complete()
            consumed += 1
        if aborted and consumed == n_chunks and not producing:
            break
        if t > 20000:
            raise RuntimeError("no progress")
    for _, s, _ in sorted(in_flight):
        full[s].complete()
    drain_ok = all(full[proto.stage(j, R)].passes(proto.drain(j, R)) for j in range(max(0, issued - R), issued))
    return overlap, drain_ok


@pytest.mark.parametrize("kernel", sorted(SOURCES))
@pytest.mark.parametrize("R", [2, 3])
def test_abort_never_refills_a_stage_with_a_copy_in_flight(kernel, R):
    """The kernels release a stage only after its copy landed, so after an
    abort no second copy enters a stage whose copy is still in flight, and
    the drain covers every copy; releasing skipped stages (the planted
    mistake) lets the producer refill them."""
    p = protocol_of(kernel)
    assert release_is_guarded(kernel)
    for seed in range(300):
        overlap, drain_ok = run_abort(p, R, 40, seed, abort_at=seed % 23, guarded=True)
        assert not overlap and drain_ok, (kernel, R, seed)
    assert any(run_abort(p, R, 40, seed, abort_at=seed % 23, guarded=False)[0] for seed in range(300))


def _broken(p, **repl):
    return Protocol(repl.get("producer", p.producer), repl.get("consumer", p.consumer),
                    repl.get("drain", p.drain), p.stage)


@pytest.mark.parametrize("mistake", [
    dict(producer=lambda i, R: (i // R) & 1),             # waits for the phase it is about to fill
    dict(producer=lambda i, R: 1 - ((i // R - 1) & 1)),   # opposite parity: passes two phases early
    dict(consumer=lambda i, R: 1 - ((i // R) & 1)),       # reads before the copy lands
    dict(drain=lambda i, R: 1 - ((i // R) & 1)),          # drain waits for a phase that never comes
])
def test_the_check_catches_a_wrong_parity(mistake):
    """Each planted mistake gives a wrong read, a hang or a drain wait that
    would never end, for at least one seed."""
    p = _broken(protocol_of("k_sparse_decode"), **mistake)
    caught = 0
    for seed in range(100):
        try:
            reads, drain_ok = run(p, 2, 40, seed, abort_at=None if seed % 2 else 20)
            caught += any(i != c for i, c in reads) or not drain_ok
        except RuntimeError:                                # the parity never comes round again
            caught += 1
    assert caught > 0
