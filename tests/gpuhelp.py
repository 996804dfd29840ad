"""Helpers of the GPU tests: device copies of a seeded case, thin wrappers
that call the C ABI, and the comparison rules against the oracle."""
from __future__ import annotations

import numpy as np
import torch

from kv_cache_page_build_b300 import kvr, synth

# attention tolerance of the decode path against the fp64 oracle (bf16 inputs)
ATOL = 2e-3
REL_L2 = 1e-3


def t16(a: np.ndarray) -> torch.Tensor:
    """bf16 bit patterns (uint16) -> int16 device tensor holding the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits_to_f64(bits(t))


class DevCase:
    def __init__(self, case: synth.Case):
        wl = case.wl
        self.case = case
        self.wl = wl
        self.k_pool = t16(case.k_pool)
        self.v_pool = t16(case.v_pool)
        self.page_table = torch.from_numpy(case.page_table).cuda()
        self.q = t16(case.q)
        self.dims = kvr.kvr_dims(**wl.dims())
        self.summ = None

    def summaries(self):
        if self.summ is None:
            wl = self.wl
            self.summ = torch.empty((wl.batch, wl.n_kv_heads, wl.n_pages, 2, wl.head_dim), dtype=torch.int16,
                                    device="cuda")
            kvr.kvr_build_summaries(self.dims, self.k_pool, self.page_table, self.summ)
        return self.summ


def workspace(d, top_k, op) -> torch.Tensor:
    n = kvr.kvr_workspace_size(d, top_k, op)
    assert n > 0
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def select(dc: DevCase, q=None, top_k=None, ws=None):
    wl = dc.wl
    k = top_k or wl.top_k
    q = dc.q if q is None else q
    sel = torch.empty((wl.batch, wl.n_kv_heads, k), dtype=torch.int32, device="cuda")
    sel_phys = torch.empty_like(sel)
    scores = torch.empty((wl.batch, wl.n_kv_heads, wl.n_pages), dtype=torch.float32, device="cuda")
    sel.fill_(-7)                      # poison: every output element must be written
    sel_phys.fill_(-7)
    scores.fill_(float("nan"))
    ws = workspace(dc.dims, k, kvr.KVR_OP_SELECT) if ws is None else ws
    kvr.kvr_select_pages(dc.dims, q, dc.summaries(), dc.page_table, k, sel, sel_phys, scores, ws, ws.numel())
    return sel, sel_phys, scores


def attention(dc: DevCase, sel_phys, q=None, top_k=None, scale=0.0, ws=None):
    wl = dc.wl
    k = top_k or wl.top_k
    q = dc.q if q is None else q
    out = torch.full((wl.batch, wl.n_q_heads, wl.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    ws = workspace(dc.dims, k, kvr.KVR_OP_ATTN) if ws is None else ws
    kvr.kvr_sparse_decode_attn(dc.dims, q, dc.k_pool, dc.v_pool, sel_phys, k, scale, out, ws, ws.numel())
    return out


def attn_errors(gpu: np.ndarray, ref: np.ndarray):
    d = gpu.astype(np.float64) - ref
    return float(np.abs(d).max()), float(np.linalg.norm(d) / np.linalg.norm(ref))


def assert_attn_close(gpu, ref):
    mx, rel = attn_errors(np.asarray(gpu), ref)
    assert mx <= ATOL and rel <= REL_L2, f"max-abs {mx:.3g}, rel-L2 {rel:.3g}"
    return mx, rel


def score_tolerance(q_bits: np.ndarray, kmin: np.ndarray, kmax: np.ndarray, G: int) -> np.ndarray:
    """Bound on |fp32 score - exact score| for the kernel's summation: each
    page score is a sum of at most 8 + log2(G) + 4 rounded additions over terms
    whose magnitudes sum to at most A = sum_h sum_c |q_hc| max(|kmin_c|, |kmax_c|);
    the error of such a sum is at most depth * 2^-24 * A, then divided by G."""
    B, Hq, D = q_bits.shape
    H = kmin.shape[1]
    qa = np.abs(synth.bf16_bits_to_f64(q_bits)).reshape(B, H, G, D)
    ka = np.maximum(np.abs(kmin), np.abs(kmax))                       # [B][H][N][D]
    A = np.einsum("bhjd,bhnd->bhn", qa, ka)
    depth = 8 + int(np.log2(G)) + 4
    return depth * 2.0 ** -24 * A / G + 1e-30
