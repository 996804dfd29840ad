"""Sensitivity of the oracle's pins: each plausible mistake, planted in the
oracle on the CPU (a wrapper around the real function), makes at least one
pin of tests/test_oracle_pins.py fail.  CPU only."""
import inspect

import numpy as np
import pytest

import oracle
import oracle.oracle as om
from tests import test_oracle_pins as pins

REAL = {name: getattr(om, name) for name in ("summaries", "scores", "topk", "attention", "group_cosine",
                                             "multi_query_step")}
PIN_TESTS = [f for name, f in inspect.getmembers(pins, inspect.isfunction)
             if name.startswith("test_") and "golden" not in name and "kv_cache_size" not in name]


def _swap_minmax(*a, **k):
    kmin, kmax = REAL["summaries"](*a, **k)
    return kmax, kmin


def _one_token_summary(k_pool, page_table, n_kv_heads=None, seq_len=None):
    first = np.repeat(np.asarray(k_pool)[:, :1], np.asarray(k_pool).shape[1], axis=1)
    return REAL["summaries"](first, page_table, n_kv_heads, seq_len=seq_len)


def _dropped_term(q, kmin, kmax):
    q = np.array(q, copy=True)
    q[..., -1] = 0                                  # the last channel never counts
    return REAL["scores"](q, kmin, kmax)


def _sum_not_mean(q, kmin, kmax):
    G = np.asarray(q).shape[1] // np.asarray(kmin).shape[1]
    return REAL["scores"](q, kmin, kmax) * G


def _group_map(q, kmin, kmax):
    return REAL["scores"](np.roll(np.asarray(q), 1, axis=1), kmin, kmax)   # head h scored with head h-1's query


def _ties_to_higher(s, k, n_valid=None):
    s = np.asarray(s)
    n = s.shape[-1]
    sel = REAL["topk"](s[..., ::-1], k, n_valid)
    return np.sort(np.where(sel >= 0, n - 1 - sel, sel), axis=-1).astype(np.int32)


def _unsorted(s, k, n_valid=None):
    sel = REAL["topk"](s, k, n_valid)
    vals = np.take_along_axis(np.asarray(s), np.maximum(sel, 0), axis=-1)
    return np.take_along_axis(sel, np.argsort(-vals, axis=-1, kind="stable"), axis=-1)


def _wrong_scale(q, k_pool, v_pool, page_table, sel, scale=None, seq_len=None):
    D = np.asarray(q).shape[-1]
    return REAL["attention"](q, k_pool, v_pool, page_table, sel, 2 * (scale or 1 / np.sqrt(D)), seq_len)


def _v_from_k(q, k_pool, v_pool, page_table, sel, scale=None, seq_len=None):
    return REAL["attention"](q, k_pool, k_pool, page_table, sel, scale, seq_len)


def _head_map(q, k_pool, v_pool, page_table, sel, scale=None, seq_len=None):
    out = REAL["attention"](np.roll(np.asarray(q), 1, axis=1), k_pool, v_pool, page_table, sel, scale, seq_len)
    return np.roll(out, -1, axis=1)                 # query head h attends with KV head of h+1's group


def _cosine_without_norms(q_t, q_prev, n_kv_heads):
    x, y = pins.f(q_t), pins.f(q_prev)
    B, Hq, _ = x.shape
    return (x * y).sum(-1).reshape(B, n_kv_heads, Hq // n_kv_heads).mean(-1)


def _lengths_off_by_one(k_pool, page_table, n_kv_heads=None, seq_len=None):
    return REAL["summaries"](k_pool, page_table, n_kv_heads,
                             seq_len=None if seq_len is None else np.asarray(seq_len) - 1)


def _causal_one_late(qs, k_pool, v_pool, page_table, n_kv_heads, top_k, seq_len, scale=None, summ=None):
    sel, s, _ = REAL["multi_query_step"](qs, k_pool, v_pool, page_table, n_kv_heads, top_k, seq_len, scale, summ)
    T = np.asarray(qs).shape[1]
    lens = np.asarray(seq_len, dtype=np.int32)
    out = np.stack([REAL["attention"](np.asarray(qs)[:, t], k_pool, v_pool, page_table, sel, scale,
                                      np.minimum(lens, lens - T + t + 2)) for t in range(T)], axis=1)
    return sel, s, out                               # query tau also sees token tau + 1


def _last_query_selects(qs, k_pool, v_pool, page_table, n_kv_heads, top_k, seq_len, scale=None, summ=None):
    qs = np.asarray(qs)
    T = qs.shape[1]
    last = np.repeat(qs[:, -1:], T, axis=1)
    sel, s, _ = REAL["multi_query_step"](last, k_pool, v_pool, page_table, n_kv_heads, top_k, seq_len, scale,
                                         summ)
    out = np.stack([REAL["attention"](qs[:, t], k_pool, v_pool, page_table, sel, scale,
                                      np.asarray(seq_len) - T + t + 1) for t in range(T)], axis=1)
    return sel, s, out


MUTATIONS = {
    "min/max swapped": ("summaries", _swap_minmax),
    "summary of the first token only": ("summaries", _one_token_summary),
    "a channel dropped from the score": ("scores", _dropped_term),
    "group score summed, not averaged": ("scores", _sum_not_mean),
    "query heads mapped to the wrong KV head in the score": ("scores", _group_map),
    "ties to the higher page id": ("topk", _ties_to_higher),
    "selection not sorted by page id": ("topk", _unsorted),
    "attention scale doubled": ("attention", _wrong_scale),
    "V read from the K pool": ("attention", _v_from_k),
    "query heads mapped to the wrong KV head in attention": ("attention", _head_map),
    "cosine without the norms": ("group_cosine", _cosine_without_norms),
    "written tokens counted one short": ("summaries", _lengths_off_by_one),
    "several queries: causal limit one token late": ("multi_query_step", _causal_one_late),
    "several queries: selection from the last query only": ("multi_query_step", _last_query_selects),
}


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(mutation, monkeypatch):
    name, fake = MUTATIONS[mutation]
    monkeypatch.setattr(oracle, name, fake)
    monkeypatch.setattr(om, name, fake)
    failed = []
    for t in PIN_TESTS:
        try:
            t()
        except AssertionError:                      # a pin's check, not a crash, must catch it
            failed.append(t.__name__)
    assert failed, f"no pin catches: {mutation}"


def test_unmutated_oracle_passes_every_pin():
    for t in PIN_TESTS:
        t()
