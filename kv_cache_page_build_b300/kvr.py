"""ctypes binding of libkvr (the C ABI declared in include/kvr.h).

Argument marshalling only: every function here forwards to the entry point of
the same name in ``libkvr.so``; all work runs in the library's CUDA kernels.
Tensors are passed as torch tensors (device or pinned host memory, as the
header states) or raw integer addresses; ``stream`` defaults to torch's
current CUDA stream.  A non-zero return code raises :class:`KvrError`.

There is no fallback: if ``libkvr.so`` has not been built, importing this
module raises.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libkvr.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "kvr.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -m kv_cache_page_build_b300.build`")

_lib = ctypes.CDLL(LIB_PATH)


def _header_constants():
    out = {}
    with open(HEADER) as f:
        for m in re.finditer(r"#define\s+(KVR_\w+)\s+\(?(-?(?:0x)?[0-9a-fA-F]+)u?\)?", f.read()):
            out[m.group(1)] = int(m.group(2), 0)
    return out


globals().update(_header_constants())


class kvr_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("batch", "n_q_heads", "n_kv_heads", "head_dim", "page_size", "n_pages", "n_phys_pages")]


class kvr_spec_state(ctypes.Structure):
    _fields_ = [("q_prev", ctypes.c_void_p), ("sel_prev", ctypes.c_void_p), ("step", ctypes.c_int32)]


class kvr_host_kv(ctypes.Structure):
    _fields_ = [("k_host", ctypes.c_void_p), ("v_host", ctypes.c_void_p)]


class kvr_working_set(ctypes.Structure):
    _fields_ = [("k_slots", ctypes.c_void_p), ("v_slots", ctypes.c_void_p),
                ("page2slot", ctypes.c_void_p), ("slot2page", ctypes.c_void_p),
                ("n_slots", ctypes.c_int32)]


class kvr_layer(ctypes.Structure):
    _fields_ = [("st", ctypes.POINTER(kvr_spec_state)), ("q", ctypes.c_void_p), ("summ", ctypes.c_void_p),
                ("page_table", ctypes.c_void_p), ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("host", ctypes.POINTER(kvr_host_kv)), ("wset", ctypes.POINTER(kvr_working_set)),
                ("out", ctypes.c_void_p), ("corrected", ctypes.c_void_p), ("cbar_opt", ctypes.c_void_p),
                ("sel_used", ctypes.c_void_p), ("sel_used_idx", ctypes.c_void_p),
                ("n_copied_opt", ctypes.c_void_p), ("ws", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t),
                ("ev", ctypes.c_void_p * 3)]


class kvr_stand_in(ctypes.Structure):
    _fields_ = [("weights", ctypes.c_void_p), ("qkv_bytes", ctypes.c_uint64), ("post_bytes", ctypes.c_uint64),
                ("sink", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_S = ctypes.c_size_t
_F = ctypes.c_float
_D = ctypes.POINTER(kvr_dims)

_SIGS = {
    "kvr_workspace_size": (_S, [_D, _I, _I]),
    "kvr_build_summaries": (_I, [_D, _P, _P, _P, _P]),
    "kvr_select_pages": (_I, [_D, _P, _P, _P, _I, _P, _P, _P, _P, _S, _P]),
    "kvr_sparse_decode_attn": (_I, [_D, _P, _P, _P, _P, _I, _F, _P, _P, _S, _P]),
    "kvr_speculative_select": (_I, [_D, ctypes.POINTER(kvr_spec_state), _P, _P, _P, _I, _F,
                                    _P, _P, _P, _P, _P, _S, _P]),
    "kvr_speculative_step": (_I, [_D, ctypes.POINTER(kvr_spec_state), _P, _P, _P, _P, _P, _I, _F,
                                  _F, _P, _P, _P, _P, _P, _P, _S, _P]),
    "kvr_speculative_step_host": (_I, [_D, ctypes.POINTER(kvr_spec_state), _P, _P, _P, _P, _P, _I, _F,
                                       _F, _P, _P, _P, _P, _P, _P, _S, _P]),
    "kvr_speculative_step_overlap": (_I, [_D, ctypes.POINTER(kvr_spec_state), _P, _P, _P, _P, _P, _I,
                                          _F, _F, _P, _P, _P, _P, _P, _P, _S, _P, _P, _P, _P]),
    "kvr_append_kv": (_I, [_D, _P, _P, _P, _P, _P, _P, _P, _P]),
    "kvr_build_summaries_len": (_I, [_D, _P, _P, _P, _P, _P]),
    "kvr_select_pages_len": (_I, [_D, _P, _P, _P, _P, _I, _P, _P, _P, _P, _S, _P]),
    "kvr_sparse_decode_attn_len": (_I, [_D, _P, _P, _P, _P, _P, _P, _I, _F, _P, _P, _S, _P]),
    "kvr_working_set_reset": (_I, [_D, ctypes.POINTER(kvr_working_set), _P]),
    "kvr_recall_pages": (_I, [_D, ctypes.POINTER(kvr_host_kv), ctypes.POINTER(kvr_working_set),
                              _P, _P, _P, _I, _P, _P, _P]),
    "kvr_speculative_step_recall": (_I, [_D, ctypes.POINTER(kvr_spec_state), _P, _P,
                                         ctypes.POINTER(kvr_host_kv), ctypes.POINTER(kvr_working_set),
                                         _I, _F, _F, _P, _P, _P, _P, _P, _P, _P, _S, _P, _P, _P, _P]),
    "kvr_pipeline_step": (_I, [_D, _I, ctypes.POINTER(kvr_layer), ctypes.POINTER(kvr_stand_in), _I, _F, _F,
                               _P, _P, _P, ctypes.POINTER(_P)]),
    "kvr_stand_in_read": (_I, [ctypes.POINTER(kvr_stand_in), ctypes.c_uint64, ctypes.c_uint64, _P]),
    "kvr_get_status": (_I, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "kvr_stream_wait": (_I, [_P, ctypes.c_uint64]),
    "kvr_set_wait_limit": (_I, [ctypes.c_uint64]),
    "kvr_select_pages_noalloc": (_I, [_D, _P, _P, _P, _I, _P, _P, _P, _P]),
    "kvr_select_pages_multi": (_I, [_D, _P, _I, _P, _P, _P, _I, _P, _P, _P, _P, _S, _P]),
    "kvr_sparse_decode_attn_multi": (_I, [_D, _P, _I, _P, _P, _P, _P, _P, _P, _I, _F, _P, _I, _P, _S, _P]),
    "kvr_error_string": (ctypes.c_char_p, [_I]),
    "kvr_kv_bytes": (ctypes.c_uint64, [ctypes.c_int64] * 5),
}

for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class KvrError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {_lib.kvr_error_string(code).decode()} ({code})")


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


_torch_c = None


def _stream(s):
    """The raw cudaStream_t of `s`; None means torch's current stream on the
    current device (read through torch's raw-stream accessor, which costs a
    fraction of building a Stream object on every call)."""
    global _torch_c
    if s is None:
        if _torch_c is None:
            import torch
            _torch_c = torch._C
        return _torch_c._cuda_getCurrentRawStream(_torch_c._cuda_getDevice())
    if isinstance(s, int):
        return s
    return getattr(s, "cuda_stream", s)


def _check(rc, where):
    if rc != 0:
        raise KvrError(rc, where)
    return rc


def dims(batch, n_q_heads, n_kv_heads, head_dim, page_size, n_pages, n_phys_pages) -> kvr_dims:
    return kvr_dims(batch, n_q_heads, n_kv_heads, head_dim, page_size, n_pages, n_phys_pages)


def _d(d):
    return ctypes.byref(d if isinstance(d, kvr_dims) else kvr_dims(**d))


def kvr_workspace_size(d, top_k, op) -> int:
    return int(_lib.kvr_workspace_size(_d(d), int(top_k), int(op)))


def kvr_build_summaries(d, k_pool, page_table, summ, stream=None):
    return _check(_lib.kvr_build_summaries(_d(d), _ptr(k_pool), _ptr(page_table), _ptr(summ),
                                           _stream(stream)), "kvr_build_summaries")


def kvr_select_pages(d, q, summ, page_table, top_k, sel, sel_phys, scores_opt, ws, ws_bytes, stream=None):
    return _check(_lib.kvr_select_pages(_d(d), _ptr(q), _ptr(summ), _ptr(page_table), int(top_k),
                                        _ptr(sel), _ptr(sel_phys), _ptr(scores_opt), _ptr(ws),
                                        int(ws_bytes), _stream(stream)), "kvr_select_pages")


def kvr_sparse_decode_attn(d, q, k_pool, v_pool, sel_phys, top_k, scale, out, ws, ws_bytes, stream=None):
    return _check(_lib.kvr_sparse_decode_attn(_d(d), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(sel_phys),
                                              int(top_k), float(scale), _ptr(out), _ptr(ws), int(ws_bytes),
                                              _stream(stream)), "kvr_sparse_decode_attn")


def kvr_speculative_select(d, st, q_t, summ, page_table, top_k, tau, corrected, cbar_opt, sel_used,
                           sel_used_phys, ws, ws_bytes, stream=None):
    return _check(_lib.kvr_speculative_select(_d(d), ctypes.byref(st), _ptr(q_t), _ptr(summ),
                                              _ptr(page_table), int(top_k), float(tau), _ptr(corrected),
                                              _ptr(cbar_opt), _ptr(sel_used), _ptr(sel_used_phys), _ptr(ws),
                                              int(ws_bytes), _stream(stream)), "kvr_speculative_select")


def kvr_speculative_step(d, st, q_t, summ, page_table, k_pool, v_pool, top_k, tau, scale, out,
                         corrected, cbar_opt, sel_used, sel_used_phys, ws, ws_bytes, stream=None):
    return _check(_lib.kvr_speculative_step(_d(d), ctypes.byref(st), _ptr(q_t), _ptr(summ), _ptr(page_table),
                                            _ptr(k_pool), _ptr(v_pool), int(top_k), float(tau), float(scale),
                                            _ptr(out), _ptr(corrected), _ptr(cbar_opt), _ptr(sel_used),
                                            _ptr(sel_used_phys), _ptr(ws), int(ws_bytes), _stream(stream)),
                  "kvr_speculative_step")


def kvr_speculative_step_host(d, st, q_host, summ, page_table, k_pool, v_pool, top_k, tau, scale, out_host,
                              corrected, cbar_opt, sel_used, sel_used_phys, ws, ws_bytes, stream=None):
    return _check(_lib.kvr_speculative_step_host(_d(d), ctypes.byref(st), _ptr(q_host), _ptr(summ),
                                                 _ptr(page_table), _ptr(k_pool), _ptr(v_pool), int(top_k),
                                                 float(tau), float(scale), _ptr(out_host), _ptr(corrected),
                                                 _ptr(cbar_opt), _ptr(sel_used), _ptr(sel_used_phys), _ptr(ws),
                                                 int(ws_bytes), _stream(stream)),
                  "kvr_speculative_step_host")


def kvr_working_set_reset(d, wset, stream=None):
    return _check(_lib.kvr_working_set_reset(_d(d), ctypes.byref(wset), _stream(stream)),
                  "kvr_working_set_reset")


def kvr_speculative_step_overlap(d, st, q_t, summ, page_table, k_pool, v_pool, top_k, tau, scale, out,
                                 corrected, cbar_opt, sel_used, sel_used_phys, ws, ws_bytes, stream,
                                 side_stream, ev_decide, ev_select):
    return _check(_lib.kvr_speculative_step_overlap(
        _d(d), ctypes.byref(st), _ptr(q_t), _ptr(summ), _ptr(page_table), _ptr(k_pool), _ptr(v_pool),
        int(top_k), float(tau), float(scale), _ptr(out), _ptr(corrected), _ptr(cbar_opt), _ptr(sel_used),
        _ptr(sel_used_phys), _ptr(ws), int(ws_bytes), _stream(stream), _stream(side_stream),
        _event(ev_decide), _event(ev_select)), "kvr_speculative_step_overlap")


def kvr_append_kv(d, k_new, v_new, page_table, seq_len, k_pool, v_pool, summ, stream=None):
    return _check(_lib.kvr_append_kv(_d(d), _ptr(k_new), _ptr(v_new), _ptr(page_table), _ptr(seq_len),
                                     _ptr(k_pool), _ptr(v_pool), _ptr(summ), _stream(stream)), "kvr_append_kv")


def kvr_build_summaries_len(d, k_pool, page_table, seq_len, summ, stream=None):
    return _check(_lib.kvr_build_summaries_len(_d(d), _ptr(k_pool), _ptr(page_table), _ptr(seq_len),
                                               _ptr(summ), _stream(stream)), "kvr_build_summaries_len")


def kvr_select_pages_len(d, q, summ, page_table, seq_len, top_k, sel, sel_phys, scores_opt, ws, ws_bytes,
                         stream=None):
    return _check(_lib.kvr_select_pages_len(_d(d), _ptr(q), _ptr(summ), _ptr(page_table), _ptr(seq_len),
                                            int(top_k), _ptr(sel), _ptr(sel_phys), _ptr(scores_opt), _ptr(ws),
                                            int(ws_bytes), _stream(stream)), "kvr_select_pages_len")


def kvr_sparse_decode_attn_len(d, q, k_pool, v_pool, page_table, seq_len, sel_phys, top_k, scale, out, ws,
                               ws_bytes, stream=None):
    return _check(_lib.kvr_sparse_decode_attn_len(_d(d), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table),
                                                  _ptr(seq_len), _ptr(sel_phys), int(top_k), float(scale),
                                                  _ptr(out), _ptr(ws), int(ws_bytes), _stream(stream)),
                  "kvr_sparse_decode_attn_len")


def kvr_recall_pages(d, host, wset, sel_new, protect, corrected, top_k, sel_slot_out, n_copied_opt,
                     stream=None):
    return _check(_lib.kvr_recall_pages(_d(d), ctypes.byref(host), ctypes.byref(wset), _ptr(sel_new),
                                        _ptr(protect), _ptr(corrected), int(top_k), _ptr(sel_slot_out),
                                        _ptr(n_copied_opt), _stream(stream)), "kvr_recall_pages")


def kvr_speculative_step_recall(d, st, q_t, summ, host, wset, top_k, tau, scale, out, corrected,
                                cbar_opt, sel_used, sel_used_slot, n_copied_opt, ws, ws_bytes,
                                stream, side_stream, ev_select, ev_recall):
    return _check(_lib.kvr_speculative_step_recall(
        _d(d), ctypes.byref(st), _ptr(q_t), _ptr(summ), ctypes.byref(host), ctypes.byref(wset),
        int(top_k), float(tau), float(scale), _ptr(out), _ptr(corrected), _ptr(cbar_opt), _ptr(sel_used),
        _ptr(sel_used_slot), _ptr(n_copied_opt), _ptr(ws), int(ws_bytes), _stream(stream),
        _stream(side_stream), _event(ev_select), _event(ev_recall)), "kvr_speculative_step_recall")


def _event(e):
    if e is None or isinstance(e, int):
        return e
    return e.cuda_event


def layer(st, q, summ, out, corrected, cbar_opt, sel_used, sel_used_idx, ws, ws_bytes, events,
          page_table=None, k_pool=None, v_pool=None, host=None, wset=None, n_copied_opt=None) -> kvr_layer:
    """A kvr_layer for kvr_pipeline_step: HBM-resident (page_table, k_pool,
    v_pool) or host-resident (host, wset); `events` are two (HBM) or three
    (host) CUDA events kept by the layer for the whole run.  The struct keeps
    st, host and wset alive; the tensors stay the caller's."""
    L = kvr_layer()
    L.st = ctypes.pointer(st)
    for name, v in (("q", q), ("summ", summ), ("page_table", page_table), ("k_pool", k_pool),
                    ("v_pool", v_pool), ("out", out), ("corrected", corrected), ("cbar_opt", cbar_opt),
                    ("sel_used", sel_used), ("sel_used_idx", sel_used_idx), ("n_copied_opt", n_copied_opt),
                    ("ws", ws)):
        setattr(L, name, _ptr(v))
    if host is not None:
        L.host = ctypes.pointer(host)
        L.wset = ctypes.pointer(wset)
    L.ws_bytes = int(ws_bytes)
    for i, e in enumerate(events):
        L.ev[i] = _event(e)
    return L


def stand_in(weights, qkv_bytes, post_bytes, sink) -> kvr_stand_in:
    """The stand-in for the rest of each layer: reads of qkv_bytes and
    post_bytes of `weights` (device), summed into `sink` (device uint32)."""
    return kvr_stand_in(_ptr(weights), int(qkv_bytes), int(post_bytes), _ptr(sink))


def kvr_stand_in_read(compute, offset, nbytes, stream=None):
    return _check(_lib.kvr_stand_in_read(ctypes.byref(compute), int(offset), int(nbytes), _stream(stream)),
                  "kvr_stand_in_read")


def kvr_pipeline_step(d, layers, compute, top_k, tau, scale, stream, side_stream, prefetch_stream, marks=None):
    """One decode step through len(layers) layers (a list of kvr_layer);
    `compute` a kvr_stand_in or None; `marks` None or
    len(layers) * KVR_PIPE_MARKS timing events, recorded once beforehand."""
    if not layers:
        raise KvrError(KVR_ERR_INVALID_ARG, "kvr_pipeline_step: no layers")
    arr = (kvr_layer * len(layers))(*layers)
    mk = None
    if marks is not None:
        if len(marks) != len(layers) * KVR_PIPE_MARKS:      # the library reads exactly that many
            raise KvrError(KVR_ERR_INVALID_ARG, f"kvr_pipeline_step: {len(marks)} marks for {len(layers)} layers")
        mk = (_P * len(marks))(*[_event(m) for m in marks])
    rc = _lib.kvr_pipeline_step(_d(d), len(layers), arr, ctypes.byref(compute) if compute is not None else None,
                                int(top_k), float(tau), float(scale), _stream(stream), _stream(side_stream),
                                _stream(prefetch_stream), mk)
    return _check(rc, "kvr_pipeline_step")


def kvr_select_pages_noalloc(d, q, summ, page_table, top_k, sel, sel_phys, scores_opt, stream=None):
    """kvr_select_pages without a caller workspace (scratch is a fixed array in
    the library; see include/kvr.h for the size limit and the sharing rule)."""
    return _check(_lib.kvr_select_pages_noalloc(_d(d), _ptr(q), _ptr(summ), _ptr(page_table), int(top_k),
                                                _ptr(sel), _ptr(sel_phys), _ptr(scores_opt), _stream(stream)),
                  "kvr_select_pages_noalloc")


def kvr_select_pages_multi(d, qs, n_query, summ, page_table, seq_len, top_k, sel, sel_phys, scores_opt, ws,
                           ws_bytes, stream=None):
    """Selection for a step of n_query query tokens per sequence (qs
    [B][T][Hq][D]; see include/kvr.h)."""
    return _check(_lib.kvr_select_pages_multi(_d(d), _ptr(qs), int(n_query), _ptr(summ), _ptr(page_table),
                                              _ptr(seq_len), int(top_k), _ptr(sel), _ptr(sel_phys),
                                              _ptr(scores_opt), _ptr(ws), int(ws_bytes), _stream(stream)),
                  "kvr_select_pages_multi")


def kvr_sparse_decode_attn_multi(d, qs, n_query, k_pool, v_pool, page_table, seq_len, sel, sel_phys, top_k,
                                 scale, out, out_dtype, ws, ws_bytes, stream=None):
    """Causal attention of n_query query tokens per sequence over the step's
    selection; out_dtype KVR_DTYPE_F32 or KVR_DTYPE_BF16."""
    return _check(_lib.kvr_sparse_decode_attn_multi(_d(d), _ptr(qs), int(n_query), _ptr(k_pool), _ptr(v_pool),
                                                    _ptr(page_table), _ptr(seq_len), _ptr(sel), _ptr(sel_phys),
                                                    int(top_k), float(scale), _ptr(out), int(out_dtype), _ptr(ws),
                                                    int(ws_bytes), _stream(stream)),
                  "kvr_sparse_decode_attn_multi")


def kvr_get_status(stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(_lib.kvr_get_status(_stream(stream), ctypes.byref(v)), "kvr_get_status")
    return int(v.value)


def kvr_stream_wait(stream=None, timeout_us: int = 0) -> bool:
    """True once the stream's work has finished, False if timeout_us passed
    first (KVR_ERR_TIMEOUT); other errors raise."""
    rc = _lib.kvr_stream_wait(_stream(stream), int(timeout_us))
    if rc == KVR_ERR_TIMEOUT:
        return False
    _check(rc, "kvr_stream_wait")
    return True


def kvr_set_wait_limit(ns: int):
    """Bound of the kernels' waits for progress, in ns (0: the default 2 s)."""
    return _check(_lib.kvr_set_wait_limit(int(ns)), "kvr_set_wait_limit")


def kvr_error_string(code: int) -> str:
    return _lib.kvr_error_string(int(code)).decode()


def kvr_kv_bytes(n_layers, n_kv_heads, head_dim, n_tokens, bytes_per_elem) -> int:
    return int(_lib.kvr_kv_bytes(n_layers, n_kv_heads, head_dim, n_tokens, bytes_per_elem))


def raw():
    """The loaded ctypes library (for tests that call entry points directly)."""
    return _lib
