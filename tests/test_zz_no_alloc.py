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
    outs = [_outputs(wl, k) for _ in range(2)]   # every buffer exists before the calls
    torch.cuda.synchronize()
    free = []
    for call, got in enumerate(outs):            # the shared scratch must be reusable call after call
        free.append(torch.cuda.mem_get_info()[0])
        kvr.kvr_select_pages_noalloc(d, q, summ, pt, k, *got)
        torch.cuda.synchronize()
        assert torch.equal(got[0], ref[0]), f"call {call}: selection differs"
        assert torch.equal(got[1], ref[1]), f"call {call}: physical ids differ"
        # same kernel and summation order as the workspace path: scores agree to the bit
        assert torch.equal(got[2], ref[2]), f"call {call}: scores differ"
    free.append(torch.cuda.mem_get_info()[0])
    # the first call on a device may load the library's device code; the
    # second call allocates nothing at all
    assert free[2] == free[1], f"free device memory changed by {free[1] - free[2]} bytes over the second call"
    assert kvr.kvr_get_status() == 0


def test_noalloc_accepts_a_problem_exactly_at_its_limit():
    """B H = 64 and N = 16383: the score rows and the per-(b, g) words fill
    the fixed array exactly (both parts multiples of 256 bytes); the result
    equals the workspace path's."""
    B, H, G, N, k = 8, 8, 4, 16383, 64
    d = kvr.kvr_dims(batch=B, n_q_heads=H * G, n_kv_heads=H, head_dim=128, page_size=16, n_pages=N,
                     n_phys_pages=B * N)
    assert kvr.kvr_workspace_size(d, k, kvr.KVR_OP_SELECT) == kvr.KVR_NOALLOC_SCRATCH_BYTES
    gen = torch.Generator(device="cuda").manual_seed(5)
    summ = torch.randn((B, H, N, 2, 128), generator=gen, device="cuda").to(torch.bfloat16).view(torch.int16)
    q = torch.randn((B, H * G, 128), generator=gen, device="cuda").to(torch.bfloat16).view(torch.int16)
    pt = torch.arange(B * N, dtype=torch.int32, device="cuda").view(B, N)
    ws = torch.zeros(kvr.KVR_NOALLOC_SCRATCH_BYTES, dtype=torch.uint8, device="cuda")

    class _W:
        batch, n_kv_heads, n_pages = B, H, N

    ref = _outputs(_W, k)
    got = _outputs(_W, k)
    kvr.kvr_select_pages(d, q, summ, pt, k, *ref, ws, ws.numel())
    kvr.kvr_select_pages_noalloc(d, q, summ, pt, k, *got)
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    assert kvr.kvr_get_status() == 0


@pytest.mark.parametrize("batch,n_pages", [(8, 16384), (64, 4096)])
def test_noalloc_rejects_problems_beyond_its_scratch(batch, n_pages):
    """One page past the limit (8 x 8 x 16384 scores: 256 bytes too many)
    and far past it are refused before anything is enqueued."""
    lib = kvr.raw()
    fake = 1 << 20                               # aligned, never dereferenced: the check comes first
    too_big = kvr.kvr_dims(batch=batch, n_q_heads=32, n_kv_heads=8, head_dim=128, page_size=16,
                           n_pages=n_pages, n_phys_pages=batch * n_pages)
    assert kvr.kvr_workspace_size(too_big, 16, kvr.KVR_OP_SELECT) > kvr.KVR_NOALLOC_SCRATCH_BYTES
    rc = lib.kvr_select_pages_noalloc(ctypes.byref(too_big), fake, fake, fake, 16, fake, None, None, None)
    assert rc == kvr.KVR_ERR_SCRATCH_LIMIT
    assert "scratch" in kvr.kvr_error_string(rc)
