"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, validates arguments before touching CUDA, and its sizing
helpers follow their definitions."""
import ctypes
import json
import os
import re

import pytest

from kv_cache_page_build_b300 import build, kvr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kvr.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvr_\w+)\s*\(", text)))


def test_library_is_current_and_exports_every_declared_symbol():
    assert build.up_to_date(), "libkvr.so is older than its sources"
    names = declared_functions()
    assert len(names) >= 12
    lib = kvr.raw()
    for n in names:
        assert hasattr(lib, n), n
        assert n in kvr._SIGS, f"binding lacks {n}"


def test_error_strings():
    for code in (kvr.KVR_OK, kvr.KVR_ERR_INVALID_ARG, kvr.KVR_ERR_UNSUPPORTED_SHAPE, kvr.KVR_ERR_ALIGN,
                 kvr.KVR_ERR_WORKSPACE, kvr.KVR_ERR_CUDA, kvr.KVR_ERR_TIMEOUT):
        assert kvr.kvr_error_string(code)
    assert "unknown" in kvr.kvr_error_string(12345)


def test_kv_bytes_matches_printed_llama65b_figure_and_overflow():
    g = json.load(open(os.path.join(GOLDEN, "kv_cache_size_llama65b.json")))
    n = kvr.kvr_kv_bytes(g["n_layers"], g["n_kv_heads"], g["head_dim"], g["n_tokens"], g["bytes_per_elem"])
    assert abs(n / 1e9 - g["stated_gb"]) <= g["stated_rounding_gb"]
    assert kvr.kvr_kv_bytes(1, 1, 1, 1, 1) == 2
    assert kvr.kvr_kv_bytes(1 << 40, 1 << 40, 1, 1, 1) == 0
    assert kvr.kvr_kv_bytes(-1, 1, 1, 1, 1) == 0


def D(**kw):
    base = dict(batch=8, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=32, n_pages=1024,
                n_phys_pages=8192)
    base.update(kw)
    return kvr.kvr_dims(**base)


def test_workspace_size_rules():
    d = D()
    sel = kvr.kvr_workspace_size(d, 64, kvr.KVR_OP_SELECT)
    att = kvr.kvr_workspace_size(d, 64, kvr.KVR_OP_ATTN)
    assert sel >= 8 * 8 * 1024 * 4 + 8 * 8 * 4
    assert att > 0                                      # a small reserved area: the split partials stay on chip
    assert kvr.kvr_workspace_size(d, 64, kvr.KVR_OP_STEP) == sel + att
    assert kvr.kvr_workspace_size(d, 2000, kvr.KVR_OP_SELECT) == 0   # k > N
    assert kvr.kvr_workspace_size(d, 64, 99) == 0
    assert kvr.kvr_workspace_size(D(head_dim=64), 64, kvr.KVR_OP_SELECT) == 0


BAD_SHAPES = [
    (dict(head_dim=64), kvr.KVR_ERR_UNSUPPORTED_SHAPE),
    (dict(n_q_heads=30), kvr.KVR_ERR_UNSUPPORTED_SHAPE),      # Hq % H != 0
    (dict(n_q_heads=24), kvr.KVR_ERR_UNSUPPORTED_SHAPE),      # G = 3
    (dict(page_size=8), kvr.KVR_ERR_UNSUPPORTED_SHAPE),
    (dict(n_pages=20000), kvr.KVR_ERR_UNSUPPORTED_SHAPE),
    (dict(batch=0), kvr.KVR_ERR_INVALID_ARG),
    (dict(n_phys_pages=-1), kvr.KVR_ERR_INVALID_ARG),
]

FAKE = 1 << 20          # a 16-byte aligned address that is never dereferenced


@pytest.mark.parametrize("kw,code", BAD_SHAPES)
def test_bad_shapes_rejected_before_launch(kw, code):
    lib = kvr.raw()
    d = D(**kw)
    assert lib.kvr_build_summaries(ctypes.byref(d), FAKE, FAKE, FAKE, None) == code
    assert lib.kvr_select_pages(ctypes.byref(d), FAKE, FAKE, FAKE, 8, FAKE, FAKE, None, FAKE, 1 << 30, None) == code
    assert lib.kvr_sparse_decode_attn(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, 8, 0.0, FAKE, FAKE, 1 << 30,
                                      None) == code


def test_bad_arguments_rejected_before_launch():
    lib = kvr.raw()
    d = D()
    big = 1 << 40
    # top_k out of range
    assert lib.kvr_select_pages(ctypes.byref(d), FAKE, FAKE, FAKE, 0, FAKE, FAKE, None, FAKE, big, None) \
        == kvr.KVR_ERR_INVALID_ARG
    assert lib.kvr_select_pages(ctypes.byref(d), FAKE, FAKE, FAKE, 1025, FAKE, FAKE, None, FAKE, big, None) \
        == kvr.KVR_ERR_UNSUPPORTED_SHAPE
    # null and misaligned pointers
    assert lib.kvr_select_pages(ctypes.byref(d), None, FAKE, FAKE, 8, FAKE, FAKE, None, FAKE, big, None) \
        == kvr.KVR_ERR_INVALID_ARG
    assert lib.kvr_select_pages(ctypes.byref(d), FAKE + 2, FAKE, FAKE, 8, FAKE, FAKE, None, FAKE, big, None) \
        == kvr.KVR_ERR_ALIGN
    assert lib.kvr_build_summaries(ctypes.byref(d), FAKE, FAKE + 4, FAKE, None) == kvr.KVR_ERR_ALIGN
    assert lib.kvr_build_summaries(None, FAKE, FAKE, FAKE, None) == kvr.KVR_ERR_INVALID_ARG
    # workspace missing or too small
    need = kvr.kvr_workspace_size(d, 64, kvr.KVR_OP_SELECT)
    assert lib.kvr_select_pages(ctypes.byref(d), FAKE, FAKE, FAKE, 64, FAKE, FAKE, None, None, need, None) \
        == kvr.KVR_ERR_WORKSPACE
    assert lib.kvr_select_pages(ctypes.byref(d), FAKE, FAKE, FAKE, 64, FAKE, FAKE, None, FAKE, need - 1, None) \
        == kvr.KVR_ERR_WORKSPACE
    need = kvr.kvr_workspace_size(d, 64, kvr.KVR_OP_ATTN)
    assert lib.kvr_sparse_decode_attn(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, 64, 0.0, FAKE, FAKE, need - 1,
                                      None) == kvr.KVR_ERR_WORKSPACE
    assert lib.kvr_sparse_decode_attn(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, 64, float("nan"), FAKE, FAKE,
                                      need, None) == kvr.KVR_ERR_INVALID_ARG


def test_speculative_and_recall_arguments_rejected_before_launch():
    lib = kvr.raw()
    d = D()
    big = 1 << 40
    st = kvr.kvr_spec_state(FAKE, FAKE, 0)
    # missing state buffers, negative step
    bad = kvr.kvr_spec_state(None, FAKE, 0)
    assert lib.kvr_speculative_select(ctypes.byref(d), ctypes.byref(bad), FAKE, FAKE, FAKE, 64, 0.8, FAKE, None,
                                      FAKE, FAKE, FAKE, big, None) == kvr.KVR_ERR_INVALID_ARG
    neg = kvr.kvr_spec_state(FAKE, FAKE, -1)
    assert lib.kvr_speculative_select(ctypes.byref(d), ctypes.byref(neg), FAKE, FAKE, FAKE, 64, 0.8, FAKE, None,
                                      FAKE, FAKE, FAKE, big, None) == kvr.KVR_ERR_INVALID_ARG
    assert lib.kvr_speculative_select(ctypes.byref(d), ctypes.byref(st), FAKE, FAKE, FAKE, 64, float("nan"),
                                      FAKE, None, FAKE, FAKE, FAKE, big, None) == kvr.KVR_ERR_INVALID_ARG
    # the full step needs sel_used_phys and a step-sized workspace
    assert lib.kvr_speculative_step(ctypes.byref(d), ctypes.byref(st), FAKE, FAKE, FAKE, FAKE, FAKE, 64, 0.8, 0.0,
                                    FAKE, FAKE, None, FAKE, None, FAKE, big, None) == kvr.KVR_ERR_INVALID_ARG
    sel_only = kvr.kvr_workspace_size(d, 64, kvr.KVR_OP_SELECT)
    assert lib.kvr_speculative_step(ctypes.byref(d), ctypes.byref(st), FAKE, FAKE, FAKE, FAKE, FAKE, 64, 0.8, 0.0,
                                    FAKE, FAKE, None, FAKE, FAKE, FAKE, sel_only, None) == kvr.KVR_ERR_WORKSPACE
    assert st.step == 0
    # working set too small for double buffering
    host = kvr.kvr_host_kv(FAKE, FAKE)
    ws = kvr.kvr_working_set(FAKE, FAKE, FAKE, FAKE, 127)
    assert lib.kvr_recall_pages(ctypes.byref(d), ctypes.byref(host), ctypes.byref(ws), FAKE, FAKE, None, 64,
                                None, None, None) == kvr.KVR_ERR_UNSUPPORTED_SHAPE
    ws.n_slots = 128
    assert lib.kvr_recall_pages(ctypes.byref(d), ctypes.byref(host), ctypes.byref(ws), FAKE, FAKE, FAKE, 64,
                                None, None, None) == kvr.KVR_ERR_INVALID_ARG   # corrected without output
    ws.k_slots = FAKE + 8
    assert lib.kvr_recall_pages(ctypes.byref(d), ctypes.byref(host), ctypes.byref(ws), FAKE, FAKE, None, 64,
                                None, None, None) == kvr.KVR_ERR_ALIGN


def test_append_and_length_arguments_rejected_before_launch():
    lib = kvr.raw()
    d = D()
    big = 1 << 40
    # append: every buffer is required, each 16-byte aligned
    args = [FAKE] * 7
    for i in range(7):
        a = list(args)
        a[i] = None
        assert lib.kvr_append_kv(ctypes.byref(d), *a, None) == kvr.KVR_ERR_INVALID_ARG
        a[i] = FAKE + 4
        assert lib.kvr_append_kv(ctypes.byref(d), *a, None) == kvr.KVR_ERR_ALIGN
    assert lib.kvr_append_kv(ctypes.byref(D(head_dim=64)), *args, None) == kvr.KVR_ERR_UNSUPPORTED_SHAPE
    # summaries, selection and attention with lengths need the lengths
    assert lib.kvr_build_summaries_len(ctypes.byref(d), FAKE, FAKE, None, FAKE, None) == kvr.KVR_ERR_INVALID_ARG
    assert lib.kvr_build_summaries_len(ctypes.byref(d), FAKE, FAKE, FAKE + 2, FAKE, None) == kvr.KVR_ERR_ALIGN
    assert lib.kvr_select_pages_len(ctypes.byref(d), FAKE, FAKE, FAKE, None, 8, FAKE, FAKE, None, FAKE, big,
                                    None) == kvr.KVR_ERR_INVALID_ARG
    assert lib.kvr_select_pages_len(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE + 4, 8, FAKE, FAKE, None, FAKE, big,
                                    None) == kvr.KVR_ERR_ALIGN
    assert lib.kvr_select_pages_len(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, 2000, FAKE, FAKE, None, FAKE, big,
                                    None) == kvr.KVR_ERR_UNSUPPORTED_SHAPE
    need = kvr.kvr_workspace_size(d, 64, kvr.KVR_OP_ATTN)
    assert lib.kvr_sparse_decode_attn_len(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, None, FAKE, 64, 0.0, FAKE, FAKE,
                                          need, None) == kvr.KVR_ERR_INVALID_ARG
    assert lib.kvr_sparse_decode_attn_len(ctypes.byref(d), FAKE, FAKE, FAKE, None, FAKE, FAKE, 64, 0.0, FAKE, FAKE,
                                          need, None) == kvr.KVR_ERR_INVALID_ARG
    assert lib.kvr_sparse_decode_attn_len(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 0.0, FAKE, FAKE,
                                          need - 1, None) == kvr.KVR_ERR_WORKSPACE


def test_pipeline_arguments_rejected_before_launch():
    """Every layer and the stand-in are checked before anything is enqueued:
    a bad second layer leaves the first layer's state untouched."""
    d = D()
    big = 1 << 40
    st0, st1 = kvr.kvr_spec_state(FAKE, FAKE, 0), kvr.kvr_spec_state(FAKE, FAKE, 0)

    def hbm_layer(st, **kw):
        args = dict(st=st, q=FAKE, summ=FAKE, out=FAKE, corrected=FAKE, cbar_opt=None, sel_used=FAKE,
                    sel_used_idx=FAKE, ws=FAKE, ws_bytes=big, events=[FAKE, FAKE],
                    page_table=FAKE, k_pool=FAKE, v_pool=FAKE)
        args.update(kw)
        return kvr.layer(**args)

    def call(layers, compute=None, marks=None, n=None, top_k=64):
        lib = kvr.raw()
        arr = (kvr.kvr_layer * max(1, len(layers)))(*layers)
        mk = None if marks is None else (ctypes.c_void_p * len(marks))(*marks)
        return lib.kvr_pipeline_step(ctypes.byref(d), len(layers) if n is None else n, arr,
                                     ctypes.byref(compute) if compute is not None else None, top_k, 0.8, 0.0,
                                     None, None, None, mk)

    good = hbm_layer(st0)
    assert call([good], n=0) == kvr.KVR_ERR_INVALID_ARG
    assert call([good], top_k=0) == kvr.KVR_ERR_INVALID_ARG
    assert call([good, hbm_layer(st1, k_pool=None)]) == kvr.KVR_ERR_INVALID_ARG
    assert call([good, hbm_layer(st1, out=FAKE + 4)]) == kvr.KVR_ERR_ALIGN
    assert call([good, hbm_layer(st1, ws_bytes=16)]) == kvr.KVR_ERR_WORKSPACE
    assert call([good, hbm_layer(kvr.kvr_spec_state(FAKE, FAKE, -1))]) == kvr.KVR_ERR_INVALID_ARG
    # a host layer needs its working set (double-buffered) and a third event
    host = kvr.kvr_host_kv(FAKE, FAKE)
    wset = kvr.kvr_working_set(FAKE, FAKE, FAKE, FAKE, 128)
    assert call([good, hbm_layer(st1, host=host, wset=wset)]) == kvr.KVR_ERR_INVALID_ARG
    assert call([good, hbm_layer(st1, host=host, wset=wset, events=[FAKE, None, FAKE])]) == kvr.KVR_ERR_INVALID_ARG
    small = kvr.kvr_working_set(FAKE, FAKE, FAKE, FAKE, 127)
    assert call([good, hbm_layer(st1, host=host, wset=small, events=[FAKE] * 3)]) == kvr.KVR_ERR_UNSUPPORTED_SHAPE
    # the stand-in: byte counts in 16-byte words, aligned weights, a sink
    assert call([good, good], compute=kvr.stand_in(FAKE, 24, 0, FAKE)) == kvr.KVR_ERR_INVALID_ARG
    assert call([good, good], compute=kvr.stand_in(FAKE, 32, 16, None)) == kvr.KVR_ERR_INVALID_ARG
    assert call([good, good], compute=kvr.stand_in(FAKE + 8, 32, 16, FAKE)) == kvr.KVR_ERR_ALIGN
    assert call([good, good], compute=kvr.stand_in(FAKE, 1 << 63, 1 << 63, FAKE)) == kvr.KVR_ERR_INVALID_ARG
    # timing marks: all n_layers * KVR_PIPE_MARKS present
    marks = [FAKE] * (2 * kvr.KVR_PIPE_MARKS)
    marks[-1] = None
    assert call([good, good], marks=marks) == kvr.KVR_ERR_INVALID_ARG
    assert st0.step == 0 and st1.step == 0


def test_stand_in_read_arguments_rejected_before_launch():
    lib = kvr.raw()
    ok = kvr.stand_in(FAKE, 32, 32, FAKE)
    assert lib.kvr_stand_in_read(None, 0, 16, None) == kvr.KVR_ERR_INVALID_ARG
    assert lib.kvr_stand_in_read(ctypes.byref(ok), 8, 16, None) == kvr.KVR_ERR_INVALID_ARG
    assert lib.kvr_stand_in_read(ctypes.byref(ok), 0, 20, None) == kvr.KVR_ERR_INVALID_ARG
    assert lib.kvr_stand_in_read(ctypes.byref(ok), 1 << 63, 1 << 63, None) == kvr.KVR_ERR_INVALID_ARG
    assert lib.kvr_stand_in_read(ctypes.byref(kvr.stand_in(FAKE, 32, 32, FAKE + 2)), 0, 16,
                                 None) == kvr.KVR_ERR_ALIGN


def test_pipeline_binding_checks_the_marks_length():
    """The library reads n_layers * KVR_PIPE_MARKS event handles; the binding
    refuses a list of another length (and an empty layer list) itself."""
    st = kvr.kvr_spec_state(FAKE, FAKE, 0)
    L = kvr.layer(st, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, 1 << 40, [FAKE, FAKE],
                  page_table=FAKE, k_pool=FAKE, v_pool=FAKE)
    with pytest.raises(kvr.KvrError):
        kvr.kvr_pipeline_step(D(), [L], None, 64, 0.8, 0.0, 0, 0, 0, marks=[FAKE] * 3)
    with pytest.raises(kvr.KvrError):
        kvr.kvr_pipeline_step(D(), [], None, 64, 0.8, 0.0, 0, 0, 0)
    assert st.step == 0


def test_host_buffer_step_arguments_rejected_before_launch():
    """kvr_speculative_step_host: its workspace holds the step's and the
    staged query's (B Hq D bf16, rounded up to 256 bytes); missing host
    buffers, state or workspace are refused before any CUDA call."""
    lib = kvr.raw()
    d = D()
    step_b = kvr.kvr_workspace_size(d, 64, kvr.KVR_OP_STEP)
    need = kvr.kvr_workspace_size(d, 64, kvr.KVR_OP_STEP_HOST)
    q_b = d.batch * d.n_q_heads * d.head_dim * 2
    assert need == step_b + (q_b + 255) // 256 * 256
    q_prev, sel_prev = FAKE, FAKE
    st = kvr.kvr_spec_state(q_prev, sel_prev, 0)

    def call(q=FAKE, out=FAKE, ws=FAKE, ws_bytes=need, state=st):
        return lib.kvr_speculative_step_host(ctypes.byref(d), ctypes.byref(state) if state else None, q, FAKE,
                                             FAKE, FAKE, FAKE, 64, 0.8, 0.0, out, FAKE, None, FAKE, FAKE, ws,
                                             ws_bytes, None)
    assert call(q=None) == kvr.KVR_ERR_INVALID_ARG
    assert call(out=None) == kvr.KVR_ERR_INVALID_ARG
    assert call(ws_bytes=need - 1) == kvr.KVR_ERR_WORKSPACE
    assert call(ws=None) == kvr.KVR_ERR_WORKSPACE
    assert call(state=None) == kvr.KVR_ERR_INVALID_ARG
    assert st.step == 0


def test_several_queries_arguments_rejected_before_launch():
    """kvr_select_pages_multi and kvr_sparse_decode_attn_multi: the query
    rows per unit (G T) must be 1, 2, 4, 8 or 16; the lengths are required,
    the logical ids too when T > 1; the output type is one of the two."""
    lib = kvr.raw()
    d = D()                                          # G = 4
    big = 1 << 40
    sel = lambda T, **kw: lib.kvr_select_pages_multi(
        ctypes.byref(kw.get("d", d)), kw.get("qs", FAKE), T, FAKE, FAKE, kw.get("lens", FAKE), 8, FAKE, FAKE, None,
        FAKE, big, None)
    assert sel(0) == kvr.KVR_ERR_INVALID_ARG
    assert sel(3) == kvr.KVR_ERR_UNSUPPORTED_SHAPE   # 12 rows
    assert sel(8) == kvr.KVR_ERR_UNSUPPORTED_SHAPE   # 32 rows
    assert sel(2, lens=None) == kvr.KVR_ERR_INVALID_ARG
    assert sel(2, qs=FAKE + 8) == kvr.KVR_ERR_ALIGN
    need = kvr.kvr_workspace_size(d, 64, kvr.KVR_OP_ATTN)

    def attn(T, sel_log=FAKE, lens=FAKE, dtype=kvr.KVR_DTYPE_F32, ws_bytes=need, dd=d):
        return lib.kvr_sparse_decode_attn_multi(ctypes.byref(dd), FAKE, T, FAKE, FAKE, FAKE, lens, sel_log, FAKE, 64,
                                                0.0, FAKE, dtype, FAKE, ws_bytes, None)
    assert attn(0) == kvr.KVR_ERR_INVALID_ARG
    assert attn(5) == kvr.KVR_ERR_UNSUPPORTED_SHAPE
    assert attn(2, sel_log=None) == kvr.KVR_ERR_INVALID_ARG       # causal limits need the logical ids
    assert attn(2, lens=None) == kvr.KVR_ERR_INVALID_ARG
    assert attn(2, dtype=2) == kvr.KVR_ERR_INVALID_ARG
    assert attn(2, sel_log=FAKE + 4) == kvr.KVR_ERR_ALIGN
    assert attn(2, ws_bytes=need - 1) == kvr.KVR_ERR_WORKSPACE
    assert attn(4, dd=D(n_q_heads=16, n_kv_heads=8), ws_bytes=need - 1) == kvr.KVR_ERR_WORKSPACE  # G 2, T 4: 8 rows
    assert attn(16, dd=D(n_q_heads=16, n_kv_heads=8)) == kvr.KVR_ERR_UNSUPPORTED_SHAPE            # 32 rows
