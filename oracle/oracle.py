"""ctypes binding and step logic of the fp64 oracle (test infrastructure only).

The arithmetic lives in ``oracle.c`` (plain C, double precision).  This file
builds it with gcc, wraps it for numpy arrays and writes out the speculative
decode logic of FreeKV (technical summary, section 2.1):

* step 0 has no previous query, so every KV head is corrected;
* for t >= 1 the group similarity C is the mean over the KV head's query
  heads of cos(q_t, q_{t-1}); a KV head whose C is lower than tau is
  corrected (it re-selects with the current query);
* the selection used at step t is the current query's selection for
  corrected heads and the previous step's selection for the others;
* the current query's selection is always computed and becomes the next
  step's "previous" selection (selection and recall run off the critical
  path every step; reuse only decides what the current attention reads).

Nothing here is imported by the CUDA path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

MARGIN = 1e-3


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, OpenMP, no
    floating-point contraction or reassociation)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i, p, d = ctypes.c_int, ctypes.c_void_p, ctypes.c_double
        L.oracle_summaries.argtypes = [i, i, i, i, i, i, p, p, p, p, p]
        L.oracle_summaries.restype = i
        L.oracle_scores.argtypes = [i, i, i, i, i, p, p, p, p]
        L.oracle_scores.restype = None
        L.oracle_topk.argtypes = [i, p, i, p]
        L.oracle_topk.restype = None
        L.oracle_topk_all.argtypes = [i, i, p, i, p, p]
        L.oracle_topk_all.restype = None
        L.oracle_attention.argtypes = [i, i, i, i, i, i, i, p, p, p, p, p, i, p, d, p]
        L.oracle_attention.restype = i
        L.oracle_group_cosine.argtypes = [i, i, i, i, p, p, p]
        L.oracle_group_cosine.restype = None
        L.oracle_set_threads.argtypes = [i]
        L.oracle_set_threads.restype = None
        L.oracle_max_threads.argtypes = []
        L.oracle_max_threads.restype = i
        _lib = L
    return _lib


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------
# primitives


def _lens(seq_len, B):
    if seq_len is None:
        return None, None
    seq_len = np.ascontiguousarray(seq_len, dtype=np.int32)
    assert seq_len.shape == (B,)
    return seq_len, seq_len.ctypes.data_as(ctypes.c_void_p)


def summaries(k_pool, page_table, n_kv_heads=None, seq_len=None):
    """(kmin, kmax), each [B][H][N][D] float64, from a [n_phys][P][H][D] bf16 pool:
    min/max over each page's written tokens (all P without seq_len [B]; NaN for
    a page with none)."""
    k_pool, kp = _c(k_pool, np.uint16)
    page_table, tp = _c(page_table, np.int32)
    n_phys, P, H, D = k_pool.shape
    B, N = page_table.shape
    seq_len, lp = _lens(seq_len, B)
    kmin = np.empty((B, H, N, D))
    kmax = np.empty((B, H, N, D))
    bad = lib().oracle_summaries(B, H, D, P, N, n_phys, kp, tp, lp,
                                 kmin.ctypes.data_as(ctypes.c_void_p),
                                 kmax.ctypes.data_as(ctypes.c_void_p))
    if bad:
        raise ValueError(f"{bad} out-of-range physical page ids")
    return kmin, kmax


def scores(q, kmin, kmax):
    """[B][H][N] float64 KV-head page scores for queries q [B][Hq][D] (bf16 bits)."""
    q, qp = _c(q, np.uint16)
    kmin, a = _c(kmin, np.float64)
    kmax, b_ = _c(kmax, np.float64)
    B, Hq, D = q.shape
    _, H, N, _ = kmin.shape
    out = np.empty((B, H, N))
    lib().oracle_scores(B, Hq, H, D, N, qp, a, b_, out.ctypes.data_as(ctypes.c_void_p))
    return out


def topk(s, k, n_valid=None):
    """Top-k page ids per row of s [..., N], ties to the lower id, sorted ascending.
    n_valid [...] (optional) limits each row to its first n_valid pages; a row
    with fewer valid pages than k selects them all and pads with -1."""
    s = np.ascontiguousarray(s, dtype=np.float64)
    lead, n = s.shape[:-1], s.shape[-1]
    units = int(np.prod(lead)) if lead else 1
    sel = np.empty(lead + (k,), dtype=np.int32)
    nv, nvp = (None, None)
    if n_valid is not None:
        nv = np.ascontiguousarray(np.broadcast_to(n_valid, lead), dtype=np.int32)
        nvp = nv.ctypes.data_as(ctypes.c_void_p)
    lib().oracle_topk_all(units, n, s.ctypes.data_as(ctypes.c_void_p), int(k), nvp,
                          sel.ctypes.data_as(ctypes.c_void_p))
    return sel


def attention(q, k_pool, v_pool, page_table, sel, scale=None, seq_len=None):
    """[B][Hq][D] float64 attention of each query head over the written tokens
    (all of them without seq_len [B]) of its KV head's selected pages."""
    q, qp = _c(q, np.uint16)
    k_pool, kp = _c(k_pool, np.uint16)
    v_pool, vp = _c(v_pool, np.uint16)
    page_table, tp = _c(page_table, np.int32)
    sel, sp = _c(sel, np.int32)
    B, Hq, D = q.shape
    n_phys, P, H, _ = k_pool.shape
    N = page_table.shape[1]
    k = sel.shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.empty((B, Hq, D))
    seq_len, lp = _lens(seq_len, B)
    bad = lib().oracle_attention(B, Hq, H, D, P, N, n_phys, qp, kp, vp, tp, sp, k, lp,
                                 float(scale), out.ctypes.data_as(ctypes.c_void_p))
    if bad:
        raise ValueError(f"{bad} out-of-range page ids")
    return out


def group_cosine(q_t, q_prev, n_kv_heads):
    """[B][H] mean over each KV head's query heads of cos(q_t, q_prev)."""
    q_t, a = _c(q_t, np.uint16)
    q_prev, b_ = _c(q_prev, np.uint16)
    B, Hq, D = q_t.shape
    out = np.empty((B, n_kv_heads))
    lib().oracle_group_cosine(B, Hq, n_kv_heads, D, a, b_, out.ctypes.data_as(ctypes.c_void_p))
    return out


# --------------------------------------------------------------------------
# one decode step and the speculative trace


def valid_pages(seq_len, page_size):
    """Pages a sequence of seq_len tokens has started: ceil(seq_len / P)."""
    return (np.asarray(seq_len, dtype=np.int64) + page_size - 1) // page_size


def select(q, k_pool, page_table, n_kv_heads, top_k, summ=None, seq_len=None):
    """Non-speculative selection: (sel [B][H][k], scores [B][H][N]); with
    seq_len [B], among each sequence's started pages only."""
    if summ is None:
        summ = summaries(k_pool, page_table, seq_len=seq_len)
    s = scores(q, *summ)
    nv = None
    if seq_len is not None:
        nv = np.repeat(valid_pages(seq_len, k_pool.shape[1])[:, None], n_kv_heads, axis=1)
    return topk(s, top_k, nv), s


def decode_step(q, k_pool, v_pool, page_table, n_kv_heads, top_k, scale=None, summ=None, seq_len=None):
    """One non-speculative decode step: returns (sel, scores, out)."""
    sel, s = select(q, k_pool, page_table, n_kv_heads, top_k, summ, seq_len)
    return sel, s, attention(q, k_pool, v_pool, page_table, sel, scale, seq_len)


def multi_query_step(qs, k_pool, v_pool, page_table, n_kv_heads, top_k, seq_len, scale=None, summ=None):
    """Several new query tokens per sequence in one step (no page treats
    this; it is the reading this oracle takes for it).  qs [B][T][Hq][D]
    bf16 bits are the queries of each sequence's last T tokens, whose K and
    V are already in the cache (seq_len [B] >= T counts them).

    * One selection per (sequence, KV head) serves the whole step: the page
      score is the mean of the upper bound over the step's T x G query rows
      (FreeKV section 2.1 averages over a KV head's query heads for group
      consistency; here the group is every query row that will read the
      pages), over the sequence's started pages.
    * Query tau (0 <= tau < T) attends causally: over the selected pages'
      tokens at positions below seq_len - T + tau + 1.

    Returns (sel [B][H][k], scores [B][H][N], out [B][T][Hq][D])."""
    qs = np.asarray(qs)
    B, T = qs.shape[0], qs.shape[1]
    seq_len = np.asarray(seq_len, dtype=np.int32)
    assert seq_len.shape == (B,) and np.all(seq_len >= T)
    if summ is None:
        summ = summaries(k_pool, page_table, seq_len=seq_len)
    s = sum(scores(qs[:, t], *summ) for t in range(T)) / T
    nv = np.repeat(valid_pages(seq_len, np.asarray(k_pool).shape[1])[:, None], n_kv_heads, axis=1)
    sel = topk(s, top_k, nv)
    out = np.stack([attention(qs[:, t], k_pool, v_pool, page_table, sel, scale, seq_len - (T - 1 - t))
                    for t in range(T)], axis=1)
    return sel, s, out


def append(k_pool, v_pool, page_table, seq_len, k_new, v_new):
    """Decode-time append ("Key-Value (KV) Cache" wiki page: each step adds
    the new token's K and V to the cache; PagedAttention fills pages in
    order): token t = seq_len[b] of sequence b goes to row t mod P of
    logical page t / P, for every KV head.  Returns new pools and lengths
    (the inputs are not modified).  k_new, v_new: [B][H][D] bf16 bits."""
    k_pool, v_pool = np.array(k_pool, copy=True), np.array(v_pool, copy=True)
    seq_len = np.array(seq_len, dtype=np.int32, copy=True)
    P = k_pool.shape[1]
    for b in range(len(seq_len)):
        t = int(seq_len[b])
        phys = int(page_table[b, t // P])
        k_pool[phys, t % P] = k_new[b]
        v_pool[phys, t % P] = v_new[b]
        seq_len[b] = t + 1
    return k_pool, v_pool, seq_len


def speculative_trace(qs, k_pool, v_pool, page_table, n_kv_heads, top_k, tau,
                      scale=None, summ=None, with_attention=True):
    """Run the speculative decode over queries qs [T][B][Hq][D].

    Returns a dict of arrays over steps: corrected [T][B][H] bool, cbar
    [T][B][H] (nan at step 0), sel_new / sel_used [T][B][H][k] and, when
    asked, out [T][B][Hq][D]."""
    if summ is None:
        summ = summaries(k_pool, page_table)
    T, B = qs.shape[0], qs.shape[1]
    H = n_kv_heads
    res = dict(corrected=np.zeros((T, B, H), bool), cbar=np.full((T, B, H), np.nan),
               sel_new=np.empty((T, B, H, top_k), np.int32),
               sel_used=np.empty((T, B, H, top_k), np.int32))
    if with_attention:
        res["out"] = np.empty((T,) + qs.shape[1:])
    prev_sel = None
    for t in range(T):
        sel_new = topk(scores(qs[t], *summ), top_k)
        if t == 0:
            corrected = np.ones((B, H), bool)
        else:
            cb = group_cosine(qs[t], qs[t - 1], H)
            res["cbar"][t] = cb
            corrected = cb < tau
        used = np.where(corrected[:, :, None], sel_new, prev_sel)
        res["corrected"][t] = corrected
        res["sel_new"][t] = sel_new
        res["sel_used"][t] = used
        if with_attention:
            res["out"][t] = attention(qs[t], k_pool, v_pool, page_table, used, scale)
        prev_sel = sel_new
    return res


# --------------------------------------------------------------------------
# acceptance predicates for the seeded generator (margins that make the
# fp32 GPU decisions provably equal to the fp64 ones)


def topk_margin(s, k):
    """S_(k) - S_(k+1) per row of s [..., N] (inf when k == N)."""
    if k >= s.shape[-1]:
        return np.full(s.shape[:-1], np.inf)
    srt = -np.sort(-s, axis=-1)
    return srt[..., k - 1] - srt[..., k]


def accept_multi_query(summ, n_kv_heads, top_k, seq_len, page_size, margin=MARGIN):
    """Predicate for synth.make_multi_queries: row b's T queries are kept
    when the step's page score (the mean over its T x G query rows, as in
    multi_query_step) has a top-k margin of at least `margin` among the
    sequence's started pages, for every KV head."""
    kmin, kmax = summ
    started = valid_pages(seq_len, page_size)

    def accept(b, q_rows):                        # q_rows [T][Hq][D] bf16 bits
        T = q_rows.shape[0]
        s = sum(scores(q_rows[t][None], kmin[b:b + 1], kmax[b:b + 1]) for t in range(T)) / T
        n = int(started[b])
        assert s.shape[1] == n_kv_heads
        return bool(np.all(topk_margin(s[..., :n], top_k) >= margin))
    return accept


def accept_single_step(top_k, margin=MARGIN):
    """Predicate for synth.make_case: row b's top-k boundary margin >= margin
    for every KV head (summaries recomputed, planted pages depend on q)."""
    def accept(case, b):
        summ = summaries(case.k_pool, case.page_table[b:b + 1])
        s = scores(case.q[b:b + 1], *summ)
        return bool(np.all(topk_margin(s, top_k) >= margin))
    return accept


def accept_trace_step(summ, n_kv_heads, top_k, tau, margin=MARGIN):
    """Predicate for synth.make_trace: at step t row b, the top-k margin of
    q_t and (t >= 1) |C - tau| are both >= margin for every KV head."""
    kmin, kmax = summ

    def accept(t, b, q_row, q_prev_row):
        s = scores(q_row[None], kmin[b:b + 1], kmax[b:b + 1])
        if not np.all(topk_margin(s, top_k) >= margin):
            return False
        cb = group_cosine(q_row[None], q_prev_row[None], n_kv_heads)
        return bool(np.all(np.abs(cb - tau) >= margin))
    return accept


def kv_cache_bytes(n_layers, n_kv_heads, head_dim, n_tokens, bytes_per_elem):
    """Bytes of a full K and V cache: 2 * layers * kv_heads * head_dim * tokens * elem."""
    return 2 * n_layers * n_kv_heads * head_dim * n_tokens * bytes_per_elem
