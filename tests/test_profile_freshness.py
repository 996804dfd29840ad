"""bench.py reports a kernel's DRAM traffic from a committed ncu record only
while the record's source hash matches the current source of what that
traffic depends on.  CPU checks of that hash: prose edits and changes
elsewhere in the library keep it; a change to the kernel's code or to the
host code that shapes its launch voids it."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _reader(edits):
    """Working-tree files with `edits` {path: (old, new)} applied."""
    def read(rel):
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        if rel in edits:
            old, new = edits[rel]
            assert old in text, (rel, old)
            text = text.replace(old, new, 1)
        return text
    return read


ATTN = "kv_cache_page_build_b300/csrc/attention.cuh"
HOST = "kv_cache_page_build_b300/csrc/kvr.cu"


def test_hash_ignores_prose_and_other_code():
    base = bench.kernel_source_hash("k_sparse_decode")
    assert bench.kernel_source_hash("k_sparse_decode", _reader({})) == base
    same = [
        {ATTN: ("#pragma once", "// a new comment line\n#pragma once")},
        {ATTN: ("#pragma once", "#pragma once\n\n\n")},
        {HOST: ("int kvr_stream_wait(", "static int unused_helper() { return 0; }\nint kvr_stream_wait(")},
        {"include/kvr.h": ("#define KVR_PIPE_MARKS 11", "#define KVR_PIPE_MARKS 12")},
    ]
    for e in same:
        assert bench.kernel_source_hash("k_sparse_decode", _reader(e)) == base, e


def test_hash_follows_the_kernel_and_its_launch():
    base = bench.kernel_source_hash("k_sparse_decode")
    changed = [
        {ATTN: ("constexpr int kAttnWarpRing = 48 * 1024;", "constexpr int kAttnWarpRing = 32 * 1024;")},
        {HOST: ("cfg.blockDim = dim3(kAttnThreads);", "cfg.blockDim = dim3(kAttnThreads + 32);")},
        {"include/kvr.h": ("#define KVR_ST_BAD_INDEX 0x1u", "#define KVR_ST_BAD_INDEX 0x10u")},
    ]
    for e in changed:
        assert bench.kernel_source_hash("k_sparse_decode", _reader(e)) != base, e


def test_committed_records_name_their_hash():
    for wl in ("llama3.1-8b-32k", "qwen3-4b-128k"):
        with open(os.path.join(ROOT, "profiles", f"k_sparse_decode_{wl}.traffic.json")) as f:
            rec = json.load(f)
        assert len(rec["source_sha256"]) == 64 and rec["dram_bytes_per_launch"] > 64 << 20
