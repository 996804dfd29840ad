"""Seeded synthetic decode-step workloads (inputs only).

This module builds the inputs that both the CUDA path and the fp64 oracle
consume: a paged bf16 K/V cache, its page table, the decode queries and the
query trace of the speculative workloads.  It holds none of the method's
arithmetic (no summaries, scores, selection or attention).  Where a workload
needs a property of the method's result (a score margin at the top-k
boundary, a cosine margin at the correction threshold), the caller passes an
``accept`` predicate and this module only redraws the query.

Shapes follow the Llama-3.1-8B and Qwen3-4B layers named on the KV Packet
review page (section 3); the query process follows the FreeKV summary
(section 2.1: adjacent decode-step queries have cosine similarity of 0.84 or
more).

Every random draw comes from its own numpy ``SeedSequence`` substream keyed by
(tensor tag, batch row, chunk / head / step, attempt), so any slice can be
regenerated alone and generation parallelises over threads.

Values are produced in float64 and rounded to bfloat16 with
round-to-nearest-even directly from float64 (no float32 double rounding).
bf16 tensors are returned as their uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Callable, Optional

import numpy as np

# substream tags
_T_TABLE, _T_K, _T_V, _T_Q, _T_PLANT_POS, _T_PLANT_NOISE = 1, 2, 3, 4, 5, 6
_T_SCALE, _T_RHO, _T_JUMPS, _T_EPS = 7, 8, 9, 10
_T_MULTI = 11

_CHUNK_PAGES = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode workload (one attention layer)."""
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    n_pages: int          # logical pages per sequence (context = n_pages * page_size)
    top_k: int            # pages selected per (sequence, KV head)
    n_planted: int = 0    # hot pages per (sequence, KV head)
    channel_scale: bool = False  # per-channel log-uniform scale in [0.25, 4]
    steps: int = 1        # decode steps (speculative trace when > 1)
    tau: Optional[float] = None  # correction threshold of the speculative mode
    n_jumps: int = 0      # topic jumps in the trace (rho = 0)
    host_resident: bool = False  # full cache lives in pinned host memory
    cache_of: Optional[int] = None  # workload id whose cache and first query it reuses
    seed: int = 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def context(self) -> int:
        return self.n_pages * self.page_size

    @property
    def n_phys_pages(self) -> int:
        return self.batch * self.n_pages

    def dims(self) -> dict:
        return dict(batch=self.batch, n_q_heads=self.n_q_heads,
                    n_kv_heads=self.n_kv_heads, head_dim=self.head_dim,
                    page_size=self.page_size, n_pages=self.n_pages,
                    n_phys_pages=self.n_phys_pages)


def _w(cid, **kw):
    return Workload(seed=1000 + cid, **kw)


WORKLOADS = {
    1: _w(1, name="tiny-4k", batch=1, n_q_heads=8, n_kv_heads=2, head_dim=128,
          page_size=16, n_pages=256, top_k=32, n_planted=4),
    2: _w(2, name="llama3.1-8b-32k", batch=8, n_q_heads=32, n_kv_heads=8,
          head_dim=128, page_size=32, n_pages=1024, top_k=64, n_planted=16),
    3: _w(3, name="qwen3-4b-128k", batch=4, n_q_heads=32, n_kv_heads=8,
          head_dim=128, page_size=32, n_pages=4096, top_k=128,
          channel_scale=True),
    4: _w(4, name="llama3.1-8b-32k-spec64", batch=8, n_q_heads=32, n_kv_heads=8,
          head_dim=128, page_size=32, n_pages=1024, top_k=64, n_planted=16,
          steps=64, tau=0.8, n_jumps=4, cache_of=2),
    5: _w(5, name="qwen3-4b-128k-host-recall32", batch=4, n_q_heads=32,
          n_kv_heads=8, head_dim=128, page_size=32, n_pages=4096, top_k=128,
          channel_scale=True, steps=32, tau=0.8, n_jumps=4, host_resident=True,
          cache_of=3),
}


# --------------------------------------------------------------------------
# rounding and random streams


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 values to bfloat16 (round to nearest, ties to even) and
    return the uint16 bit patterns.  Finite, normal-range inputs only."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m * 2**e, 0.5 <= |m| < 1
    y = np.ldexp(np.rint(m * 256.0), e - 8)  # keep 8 significant bits, RNE
    return (y.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_bits_to_f64(b) -> np.ndarray:
    """Exact widening of bf16 bit patterns."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(seed, spawn_key=tuple(int(k) for k in key)))


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


# --------------------------------------------------------------------------
# cache


@dataclasses.dataclass
class Case:
    """One workload's inputs.  Arrays are numpy; bf16 as uint16 bits.

    k_pool, v_pool : [n_phys_pages][page_size][n_kv_heads][head_dim]  (NHD pages)
    page_table     : [batch][n_pages] int32, logical page -> physical page
    q              : [batch][n_q_heads][head_dim]
    planted        : [batch][n_kv_heads][n_planted] int32 logical page ids
    k_scale/v_scale: [n_kv_heads][head_dim] float64 channel scales (or None)
    q_attempt      : [batch] int, redraw counter of each row's accepted query
    """
    wl: Workload
    k_pool: np.ndarray
    v_pool: np.ndarray
    page_table: np.ndarray
    q: np.ndarray
    planted: np.ndarray
    k_scale: Optional[np.ndarray]
    v_scale: Optional[np.ndarray]
    q_attempt: np.ndarray
    plant_noise: Optional[np.ndarray] = None  # [batch][n_kv_heads][n_planted][P][D] float64


def _channel_scales(wl: Workload):
    if not wl.channel_scale:
        return None, None
    lo, hi = np.log(0.25), np.log(4.0)
    ks = np.exp(_rng(wl.seed, _T_SCALE, 0).uniform(lo, hi, size=(wl.n_kv_heads, wl.head_dim)))
    vs = np.exp(_rng(wl.seed, _T_SCALE, 1).uniform(lo, hi, size=(wl.n_kv_heads, wl.head_dim)))
    return ks, vs


def _fill_pool(wl: Workload, tag: int, scale, page_table, pool):
    P, H, D = wl.page_size, wl.n_kv_heads, wl.head_dim
    jobs = [(b, c) for b in range(wl.batch) for c in range(0, wl.n_pages, _CHUNK_PAGES)]

    def run(job):
        b, c = job
        n = min(_CHUNK_PAGES, wl.n_pages - c)
        z = _rng(wl.seed, tag, b, c).standard_normal((n, P, H, D))
        if scale is not None:
            z *= scale[None, None, :, :]
        pool[page_table[b, c:c + n]] = f64_to_bf16_bits(z)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(run, jobs))


def _draw_q(wl: Workload, b: int, attempt: int) -> np.ndarray:
    z = _rng(wl.seed, _T_Q, b, attempt).standard_normal((wl.n_q_heads, wl.head_dim))
    return f64_to_bf16_bits(z)


def query_direction(wl: Workload, q_row_bits: np.ndarray) -> np.ndarray:
    """Per KV head, the mean of its group's query heads scaled to unit RMS per
    element: [n_kv_heads][head_dim] float64.  Used to build the planted pages
    (key = 0.8 * q_dir + 0.6 * noise has unit variance per element)."""
    qf = bf16_bits_to_f64(q_row_bits).reshape(wl.n_kv_heads, wl.group, wl.head_dim)
    qbar = qf.mean(axis=1)
    rms = np.sqrt((qbar * qbar).mean(axis=1, keepdims=True))
    return qbar / rms


def _plant(case: Case, b: int):
    wl = case.wl
    if wl.n_planted == 0:
        return
    qd = query_direction(wl, case.q[b])
    for g in range(wl.n_kv_heads):
        for i, p in enumerate(case.planted[b, g]):
            keys = 0.8 * qd[g][None, :] + 0.6 * case.plant_noise[b, g, i]
            case.k_pool[case.page_table[b, p], :, g, :] = f64_to_bf16_bits(keys)


def make_case(wl, accept: Optional[Callable[[Case, int], bool]] = None,
              max_attempts: int = 200) -> Case:
    """Build a workload's cache and single-step query.

    ``wl`` is a Workload or a workload id.  For the speculative / host
    workloads this returns the cache and first query of the workload they
    reuse.  ``accept(case, b)`` (optional) decides whether batch row ``b``'s
    query is kept; rejected rows are redrawn with the next attempt counter
    (planted pages are rebuilt from the new query with the same noise).
    """
    if isinstance(wl, int):
        wl = WORKLOADS[wl]
    if wl.cache_of is not None:
        wl = WORKLOADS[wl.cache_of]
    B, N, P, H, D = wl.batch, wl.n_pages, wl.page_size, wl.n_kv_heads, wl.head_dim
    page_table = _rng(wl.seed, _T_TABLE).permutation(B * N).astype(np.int32).reshape(B, N)
    k_scale, v_scale = _channel_scales(wl)
    k_pool = np.empty((B * N, P, H, D), dtype=np.uint16)
    v_pool = np.empty((B * N, P, H, D), dtype=np.uint16)
    _fill_pool(wl, _T_K, k_scale, page_table, k_pool)
    _fill_pool(wl, _T_V, v_scale, page_table, v_pool)

    planted = np.zeros((B, H, wl.n_planted), dtype=np.int32)
    noise = None
    if wl.n_planted:
        noise = np.empty((B, H, wl.n_planted, P, D))
        for b in range(B):
            for g in range(H):
                planted[b, g] = np.sort(_rng(wl.seed, _T_PLANT_POS, b, g).choice(N, wl.n_planted, replace=False))
                noise[b, g] = _rng(wl.seed, _T_PLANT_NOISE, b, g).standard_normal((wl.n_planted, P, D))

    q = np.stack([_draw_q(wl, b, 0) for b in range(B)])
    case = Case(wl, k_pool, v_pool, page_table, q, planted, k_scale, v_scale,
                np.zeros(B, dtype=np.int64), noise)
    for b in range(B):
        _plant(case, b)
        if accept is None:
            continue
        while not accept(case, b):
            case.q_attempt[b] += 1
            if case.q_attempt[b] >= max_attempts:
                raise RuntimeError(f"{wl.name}: no accepted query for row {b} in {max_attempts} draws")
            case.q[b] = _draw_q(wl, b, int(case.q_attempt[b]))
            _plant(case, b)
    return case


def host_hnd(case: Case):
    """The cache in the host (HND) layout: [batch][n_kv_heads][n_pages][page_size][head_dim],
    i.e. one contiguous P x D block per (sequence, KV head, logical page)."""
    wl = case.wl
    out = []
    for pool in (case.k_pool, case.v_pool):
        logical = pool[case.page_table.reshape(-1)].reshape(
            wl.batch, wl.n_pages, wl.page_size, wl.n_kv_heads, wl.head_dim)
        out.append(np.ascontiguousarray(logical.transpose(0, 3, 1, 2, 4)))
    return out[0], out[1]


# --------------------------------------------------------------------------
# speculative query trace


@dataclasses.dataclass
class Trace:
    """q: [steps][batch][n_q_heads][head_dim] bf16 bits; rho: [steps] (rho[0] unused);
    jumps: sorted step ids with rho = 0; attempts: [steps][batch] redraw counters."""
    q: np.ndarray
    rho: np.ndarray
    jumps: np.ndarray
    attempts: np.ndarray


def trace_rhos(wl: Workload) -> tuple[np.ndarray, np.ndarray]:
    """Per-step AR(1) coefficient: U[0.84, 0.98] with probability 0.9, else
    U[0.60, 0.84]; ``n_jumps`` seed-chosen steps in [1, steps) get rho = 0."""
    T = wl.steps
    rho = np.zeros(T)
    for t in range(1, T):
        r = _rng(wl.seed, _T_RHO, t)
        rho[t] = r.uniform(0.84, 0.98) if r.uniform() < 0.9 else r.uniform(0.60, 0.84)
    jumps = np.sort(_rng(wl.seed, _T_JUMPS).choice(np.arange(1, T), wl.n_jumps, replace=False)) if wl.n_jumps else np.zeros(0, np.int64)
    rho[jumps] = 0.0
    return rho, jumps


def make_trace(wl, case: Case,
               accept: Optional[Callable[[int, int, np.ndarray, np.ndarray], bool]] = None,
               max_attempts: int = 200) -> Trace:
    """AR(1) query trace q_t = rho_t * q_{t-1} + sqrt(1 - rho_t^2) * eps_t.

    The process runs in float64 from the first query (the cache workload's
    accepted query); each step is handed out rounded to bf16.  ``accept(t, b,
    q_t_row, q_prev_row)`` (optional) may reject row ``b`` of step ``t``; the
    innovation eps_t of that row is then redrawn, so earlier steps never
    change.
    """
    if isinstance(wl, int):
        wl = WORKLOADS[wl]
    T, B = wl.steps, case.wl.batch
    rho, jumps = trace_rhos(wl)
    qs = np.empty((T,) + case.q.shape, dtype=np.uint16)
    attempts = np.zeros((T, B), dtype=np.int64)
    qs[0] = case.q
    state = bf16_bits_to_f64(case.q)
    for t in range(1, T):
        a = rho[t]
        c = np.sqrt(max(0.0, 1.0 - a * a))
        for b in range(B):
            n = 0
            while True:
                eps = _rng(wl.seed, _T_EPS, t, b, n).standard_normal(state.shape[1:])
                cand = a * state[b] + c * eps
                bits = f64_to_bf16_bits(cand)
                if accept is None or accept(t, b, bits, qs[t - 1, b]):
                    break
                n += 1
                if n >= max_attempts:
                    raise RuntimeError(f"{wl.name}: no accepted innovation at step {t} row {b}")
            attempts[t, b] = n
            state[b] = cand
            qs[t, b] = bits
    return Trace(qs, rho, jumps, attempts)


def make_multi_queries(case: Case, T: int, accept: Optional[Callable[[int, np.ndarray], bool]] = None,
                       rho: float = 0.9, max_attempts: int = 200) -> np.ndarray:
    """T query tokens per sequence for one step of several queries: an AR(1)
    run q_tau = rho q_{tau-1} + sqrt(1 - rho^2) eps_tau from the case's
    query, in float64, each token handed out rounded to bf16.
    ``accept(b, rows)`` (rows [T][Hq][D] bits, optional) may reject row b,
    whose innovations are then redrawn with the next attempt counter.
    Returns [B][T][Hq][D] bf16 bits."""
    wl = case.wl
    c = np.sqrt(1.0 - rho * rho)
    out = np.empty((wl.batch, T) + case.q.shape[1:], dtype=np.uint16)
    for b in range(wl.batch):
        n = 0
        while True:
            state = bf16_bits_to_f64(case.q[b])
            rows = []
            for t in range(T):
                state = rho * state + c * _rng(wl.seed, _T_MULTI, b, t, n).standard_normal(state.shape)
                rows.append(f64_to_bf16_bits(state))
            rows = np.stack(rows)
            if accept is None or accept(b, rows):
                break
            n += 1
            if n >= max_attempts:
                raise RuntimeError(f"{wl.name}: no accepted queries for row {b} in {max_attempts} draws")
        out[b] = rows
    return out


def custom(name="custom", **kw) -> Workload:
    """A small workload for tests (fields as in Workload; seed defaults to 7)."""
    kw.setdefault("seed", 7)
    return Workload(name=name, **kw)
