"""The allocation-free selection entry point, for callers that cannot
allocate device memory (an engine plugin limited to the buffers it is handed,
a serving loop that forbids allocation after warm-up, a foreign-language
caller without the process's allocator).  It must return exactly what the
workspace-based kvr_select_pages returns, call after call, while its scratch
lives in a fixed array inside the library.

This file is collected last on purpose, and builds its own inputs so it also
passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from kv_cache_page_build_b300 import kvr, synth

pytestmark = pytest.mark.gpu


def _device_case(**kw):
    wl = synth.custom(**kw)
    case = synth.make_case(wl)
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    d = kvr.kvr_dims(**wl.dims())
    k_pool = to(case.k_pool.view(np.int16))
    pt = to(case.page_table)
    summ = torch.empty((wl.batch, wl.n_kv_heads, wl.n_pages, 2, wl.head_dim), dtype=torch.int16, device="cuda")
    kvr.kvr_build_summaries(d, k_pool, pt, summ)
    return wl, d, to(case.q.view(np.int16)), summ, pt


def _outputs(wl, k):
    sel = torch.full((wl.batch, wl.n_kv_heads, k), -7, dtype=torch.int32, device="cuda")
    return sel, torch.full_like(sel, -7), torch.full((wl.batch, wl.n_kv_heads, wl.n_pages), float("nan"),
                                                     dtype=torch.float32, device="cuda")


@pytest.mark.parametrize("shape", [
    dict(batch=8, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=32, n_pages=1024, top_k=64),
    dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=16, n_pages=333, top_k=29),
])
def test_noalloc_selection_equals_workspace_selection_twice(shape):
    wl, d, q, summ, pt = _device_case(**shape)
    k = wl.top_k
    ws = torch.zeros(kvr.kvr_workspace_size(d, k, kvr.KVR_OP_SELECT), dtype=torch.uint8, device="cuda")
    ref = _outputs(wl, k)
    kvr.kvr_select_pages(d, q, summ, pt, k, *ref, ws, ws.numel())
    for call in range(2):                      # the shared scratch must be reusable call after call
        got = _outputs(wl, k)
        kvr.kvr_select_pages_noalloc(d, q, summ, pt, k, *got)
        torch.cuda.synchronize()
        assert torch.equal(got[0], ref[0]), f"call {call}: selection differs"
        assert torch.equal(got[1], ref[1]), f"call {call}: physical ids differ"
        # same kernel and summation order as the workspace path: scores agree to the bit
        assert torch.equal(got[2], ref[2]), f"call {call}: scores differ"
    assert kvr.kvr_get_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = kvr.raw()
    fake = 1 << 20                               # aligned, never dereferenced: the check comes first
    too_big = kvr.kvr_dims(batch=64, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=32, n_pages=4096,
                           n_phys_pages=64 * 4096)
    assert 64 * 8 * 4096 * 4 > kvr.KVR_NOALLOC_SCRATCH_BYTES
    rc = lib.kvr_select_pages_noalloc(ctypes.byref(too_big), fake, fake, fake, 16, fake, None, None, None)
    assert rc == kvr.KVR_ERR_SCRATCH_LIMIT
    assert "scratch" in kvr.kvr_error_string(rc)
