"""Model check of the multi-layer pipeline's stream schedule (CPU only).

The operations kvr_pipeline_step enqueues per layer -- kernel launches, event
records and stream waits, on the main, side and prefetch streams -- are read
from its source in csrc/kvr.cu, unrolled over layers and decode steps in
enqueue order, and turned into a happens-before graph (each stream runs its
operations in order; a wait orders everything after it behind the latest
record of its event at enqueue time).  Each kernel is given the buffers it
reads and writes.  Two accesses to one buffer, at least one a write, must be
ordered, except where the kernels make them disjoint: the units of a step
are split into reused and corrected ones, and a recall writes only slots
that the running attention does not read.  The check passes on the schedule
as written and fails on schedules with a wait or a record moved or dropped.
"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _code(text):
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def _balanced(code, i, open_ch, close_ch):
    """Index just past the bracket matching code[i] == open_ch."""
    depth = 0
    while True:
        depth += {open_ch: 1, close_ch: -1}.get(code[i], 0)
        i += 1
        if depth == 0:
            return i


def _statements(code):
    """The KVR_TRY(...) statements of `code`, in order, as their inner text."""
    out = []
    for m in re.finditer(r"KVR_TRY\(", code):
        end = _balanced(code, m.end() - 1, "(", ")")
        out.append(code[m.end():end - 1].strip())
    return out


def _classify(stmt):
    """One operation (kind, stream, detail) of a statement."""
    args = lambda s: [a.strip() for a in s[s.index("(") + 1:s.rindex(")")].split(",")]
    name = stmt[:stmt.index("(")].strip()
    a = args(stmt)
    if name == "mark":
        return ("mark", a[2], None)
    if name == "record":
        return ("record", a[1], int(re.search(r"ev\[(\d)\]", a[0]).group(1)))
    if name == "wait":
        return ("wait", a[0], int(re.search(r"ev\[(\d)\]", a[1]).group(1)))
    if name == "launch_stand_in":
        return ("kernel", a[-1], "stand_in")
    if name == "launch_spec_decide":
        return ("kernel", a[-1], "decide")
    if name == "launch_select":
        part = {"kSelScores": "scores", "kSelTopk": "topk"}.get(a[-1], "select")
        return ("kernel", a[a.index("sa") + 1], part)
    if name == "spec_select_impl":
        stream = a[a.index("L.ws") + 1]
        # with the early-start words (HBM): the whole selection of the step,
        # the attention after it reading the reused units' ids early
        return ("kernel", stream, "spec_step_select" if "aw.ready" in a else "spec_select")
    if name == "launch_recall":
        return ("kernel", a[-2], {"2": "recall_corrected", "1": "recall_prefetch"}[a[-1]])
    if name == "launch_attn":
        stream = a[a.index("L.out") + 1]
        if "L.corrected" not in a:
            return ("kernel", stream, "attn_all")
        mode = a[a.index("L.corrected") + 1]
        return ("kernel", stream, {"1": "attn_reused", "2": "attn_corrected"}[mode])
    raise AssertionError(f"unknown statement {stmt!r}")


def pipeline_schedule():
    """(prologue, HBM branch, host branch, epilogue) of one layer, read from
    kvr_pipeline_step."""
    code = _code(open(os.path.join(ROOT, "kv_cache_page_build_b300", "csrc", "kvr.cu")).read())
    start = code.index("int kvr_pipeline_step(")
    body = code[start:code.index("#undef KVR_TRY", start)]
    loop = body[body.index("for (int l = 0; l < n_layers; ++l) {"):]
    i_if = loop.index("if (!L.host) {")
    i_hbm = i_if + len("if (!L.host) ")
    e_hbm = _balanced(loop, i_hbm, "{", "}")
    rest = loop[e_hbm:].lstrip()
    assert rest.startswith("else {")
    i_host = e_hbm + loop[e_hbm:].index("{")
    e_host = _balanced(loop, i_host, "{", "}")
    parts = (loop[:i_if], loop[i_hbm:e_hbm], loop[i_host:e_host], loop[e_host:])
    return tuple([_classify(s) for s in _statements(p)] for p in parts)


# Buffers each kernel reads (R) and writes (W), per layer unless marked
# shared ("ws").  A ".r" / ".c" suffix: only the reused / corrected units of
# the step.  Constant inputs (q, summaries, pools, host cache, weights) and
# the atomically summed sink and copy counter are left out.
ACCESS = {
    "stand_in": ((), ()),
    "decide": (("q_prev", "sel_prev"), ("corrected", "cbar", "q_prev", "sel_used.r", "idx.r")),
    "select": (("corrected",), ("ws", "sel_prev", "sel_used.c", "idx.c")),
    "scores": ((), ("ws",)),
    "topk": (("corrected", "ws"), ("sel_prev", "sel_used.c", "idx.c")),
    "spec_select": (("q_prev", "sel_prev", "maps"),
                    ("ws", "corrected", "cbar", "q_prev", "sel_prev", "sel_used", "idx.r")),
    "spec_step_select": (("q_prev", "sel_prev"),
                         ("ws", "corrected", "cbar", "q_prev", "sel_prev", "sel_used", "idx")),
    "recall_corrected": (("sel_prev", "sel_used", "corrected", "maps.c"), ("maps.c", "slots.c", "idx.c")),
    "recall_prefetch": (("sel_prev", "sel_used", "corrected", "maps.r"), ("maps.r", "slots.r")),
    "attn_reused": (("corrected", "idx.r", "slots.r"), ("out.r",)),
    "attn_corrected": (("corrected", "idx.c", "slots.c"), ("out.c",)),
    # reads the early-start words in the workspace and clears them
    "attn_all": (("idx", "ws"), ("out", "ws")),
}
SHARED = {"ws"}


class Op:
    def __init__(self, idx, kind, stream, detail, layer, step):
        self.idx, self.kind, self.stream, self.detail = idx, kind, stream, detail
        self.layer, self.step = layer, step
        self.before = 0            # bitmask of operations that happen before this one


def unroll(schedule, kinds, steps, shared_events=False, join=False):
    """Enqueue `steps` pipeline steps over layers of the given kinds ("hbm" or
    "host"); returns the operations with their happens-before sets."""
    pro, hbm, host, epi = schedule
    ops, last, latest = [], {}, {}

    def add(kind, stream, detail, layer, step):
        op = Op(len(ops), kind, stream, detail, layer, step)
        if stream in last:                                   # stream order
            prev = ops[last[stream]]
            op.before |= prev.before | (1 << prev.idx)
        if kind == "wait":
            key = detail if shared_events else (layer, detail)
            if key in latest:                                # the latest record at enqueue time
                rec = ops[latest[key]]
                op.before |= rec.before | (1 << rec.idx)
        if kind == "record":
            latest[detail if shared_events else (layer, detail)] = op.idx
        last[stream] = op.idx
        ops.append(op)

    for t in range(steps):
        for l, kind in enumerate(kinds):
            for k, stream, detail in pro + (hbm if kind == "hbm" else host) + epi:
                add(k, stream, detail, l, t)
    if join:
        for l, kind in enumerate(kinds):
            if kind == "host":
                add("wait", "s", 2, l, steps)
        add("kernel", "s", "stand_in", -1, steps)            # whatever follows on the main stream
    return ops


def _accesses(op):
    reads, writes = ACCESS[op.detail]
    return [(b, False) for b in reads] + [(b, True) for b in writes]


def _disjoint(a, ba, b, bb):
    """Accesses the kernels keep apart within one step of one layer."""
    if a.step != b.step or a.layer != b.layer:
        return False
    pa = ba.split(".")[1] if "." in ba else None
    pb = bb.split(".")[1] if "." in bb else None
    if pa and pb and pa != pb:
        return True                                          # reused vs corrected units
    recall = {"recall_corrected", "recall_prefetch"}
    attn = {"attn_reused", "attn_corrected"}
    if ba.startswith("slots") and ({a.detail, b.detail} & recall) and ({a.detail, b.detail} & attn):
        return True                                          # recall writes only unprotected slots
    return False


def races(ops):
    kernels = [o for o in ops if o.kind == "kernel"]
    found = []
    for i, a in enumerate(kernels):
        for b in kernels[i + 1:]:
            ordered = (b.before >> a.idx) & 1 or (a.before >> b.idx) & 1
            if ordered:
                continue
            for ba, wa in _accesses(a):
                for bb, wb in _accesses(b):
                    if ba.split(".")[0] != bb.split(".")[0] or not (wa or wb):
                        continue
                    if ba.split(".")[0] not in SHARED and a.layer != b.layer:
                        continue
                    if _disjoint(a, ba, b, bb):
                        continue
                    found.append((a.detail, a.layer, a.step, b.detail, b.layer, b.step, ba, bb))
    return found


KINDS = [["hbm"] * 3, ["host"] * 3, ["hbm", "host", "hbm"], ["host", "hbm", "host"]]


def test_schedule_is_read_from_the_source():
    pro, hbm, host, epi = pipeline_schedule()
    kernels = lambda seq: [d for k, _, d in seq if k == "kernel"]
    assert kernels(pro) == ["stand_in"] and kernels(epi) == ["stand_in"]
    assert kernels(hbm) == ["spec_step_select", "attn_all"]
    assert all(stream == "s" for _, stream, _ in hbm)
    assert kernels(host) == ["spec_select", "recall_corrected", "recall_prefetch", "attn_reused",
                             "attn_corrected"]
    assert sum(k == "mark" for k, _, _ in pro + hbm + epi) == 11
    assert sum(k == "mark" for k, _, _ in pro + host + epi) == 11


@pytest.mark.parametrize("kinds", KINDS)
@pytest.mark.parametrize("shared_events", [False, True])
def test_no_unordered_conflicting_accesses(kinds, shared_events):
    """Three steps of three layers: every pair of conflicting accesses is
    ordered, also with one set of events shared by all layers."""
    assert races(unroll(pipeline_schedule(), kinds, 3, shared_events=shared_events)) == []


def test_join_orders_every_operation_before_what_follows():
    """With the main stream waiting on each host layer's prefetch event after
    the last step, every operation happens before what the caller enqueues
    next; without it, the last prefetches do not."""
    kinds = ["host", "hbm", "host"]
    ops = unroll(pipeline_schedule(), kinds, 2, join=True)
    final = ops[-1]
    assert all((final.before >> o.idx) & 1 for o in ops[:-1])
    ops = unroll(pipeline_schedule(), kinds, 2)
    tail = ops[-1]
    loose = [o.detail for o in ops[:-1] if not (tail.before >> o.idx) & 1 and o.kind == "kernel"]
    assert "recall_prefetch" in loose


def _mutated(drop=None, move=None, restream=None):
    pro, hbm, host, epi = pipeline_schedule()
    hbm, host = list(hbm), list(host)
    if restream:
        branch, op, stream = restream
        seq = hbm if branch == "hbm" else host
        seq[seq.index(op)] = (op[0], stream, op[2])
    if drop:
        branch, op = drop
        seq = hbm if branch == "hbm" else host
        seq.remove(op)
    if move:
        branch, op, before = move
        seq = hbm if branch == "hbm" else host
        seq.remove(op)
        seq.insert(seq.index(before), op)
    return pro, hbm, host, epi


@pytest.mark.parametrize("mutation,kinds", [
    (dict(drop=("host", ("wait", "s", 2))), ["host"] * 2),                       # no wait for last prefetch
    (dict(drop=("host", ("wait", "s", 1))), ["host"] * 2),                       # corrected heads don't wait
    (dict(restream=("hbm", ("kernel", "s", "attn_all"), "side")), ["hbm"] * 2),   # attention beside its selection
    (dict(drop=("host", ("wait", "pf", 1))), ["host"] * 2),                      # prefetch before selection
    (dict(move=("host", ("record", "side", 1), ("kernel", "side", "recall_corrected"))), ["host"] * 2),
    (dict(restream=("hbm", ("kernel", "s", "spec_step_select"), "side")), ["hbm", "host"]),  # selection off the chain
])
def test_the_check_catches_a_broken_schedule(mutation, kinds):
    assert races(unroll(_mutated(**mutation), kinds, 3)) != []
