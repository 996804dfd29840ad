// summaries.cuh -- per-page, per-channel key min/max (page summaries).
//
// The paged K cache ("Key-Value (KV) Cache" wiki page, PagedAttention) is
// reduced once per cache to one min row and one max row per (sequence, KV
// head, logical page).  The selection kernel scores pages from these rows.
//
// Work mapping: a token row of the pool holds all H heads (H * 256 bytes).
// One thread owns one 16-byte column (8 channels of one head) of one page and
// walks the page's P tokens; the min/max of bf16 values is taken in bf16
// (exact).  A 256-thread CTA covers 256 / (16 H) pages side by side, so a
// warp reads 512 contiguous bytes per token.  A thread issues its loads in
// batches of up to 16 tokens before consuming them (256 bytes in flight).
#pragma once

#include "common.cuh"

namespace kvr {

constexpr int kSumThreads = 256;

// seq_len (may be null): sequence b has written seq_len[b] tokens, so page p
// holds min(P, seq_len[b] - p P) of them; a page with none is left as is.
template <int P>
__global__ void __launch_bounds__(kSumThreads)
    k_build_summaries(const uint16_t *__restrict__ k_pool, const int32_t *__restrict__ page_table,
                      const int32_t *__restrict__ seq_len, uint16_t *__restrict__ summ, int H,
                      int N, int n_phys, int pages_per_cta) {
  const int cols = H * 16;  // 16-byte columns per token row
  const int b = blockIdx.y;
  const size_t token_stride = static_cast<size_t>(H) * kD;  // elements between tokens
  for (int idx = threadIdx.x; idx < pages_per_cta * cols; idx += kSumThreads) {
    const int pl = idx / cols;
    const int col = idx - pl * cols;
    const int p = blockIdx.x * pages_per_cta + pl;
    if (p >= N) continue;
    const int nt = seq_len ? min(P, max(0, seq_len[b] - p * P)) : P;  // written tokens
    if (nt == 0) continue;
    const int phys = page_table[static_cast<size_t>(b) * N + p];
    const int g = col >> 4, j = col & 15;
    if (phys < 0 || phys >= n_phys) {
      if (col == 0) set_status(KVR_ST_BAD_INDEX);
      continue;
    }
    const uint16_t *src =
        k_pool + (static_cast<size_t>(phys) * P * H + g) * kD + 8 * j;  // token 0
    constexpr int BT = P < 16 ? P : 16;  // tokens loaded per batch (BT * 16 B in flight)
    __nv_bfloat162 mn[4], mx[4];
#pragma unroll
    for (int t0 = 0; t0 < P; t0 += BT) {
      uint4 v[BT];
#pragma unroll
      for (int t = 0; t < BT; ++t) v[t] = ld_stream_v4(src + (t0 + t) * token_stride);
#pragma unroll
      for (int t = 0; t < BT; ++t) {
        const __nv_bfloat162 *w = reinterpret_cast<const __nv_bfloat162 *>(&v[t]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (t0 == 0 && t == 0) {
            mn[i] = mx[i] = w[i];
          } else if (t0 + t < nt) {
            mn[i] = __hmin2(mn[i], w[i]);
            mx[i] = __hmax2(mx[i], w[i]);
          }
        }
      }
    }
    uint16_t *dst = summ + ((static_cast<size_t>(b) * H + g) * N + p) * (2 * kD) + 8 * j;
    *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(mn);
    *reinterpret_cast<uint4 *>(dst + kD) = *reinterpret_cast<const uint4 *>(mx);
  }
}

// Decode-time append ("Key-Value (KV) Cache" wiki page: each decode step
// adds the new token's key and value to the cache; PagedAttention fills a
// sequence's pages in order).  One CTA per sequence b: token t = seq_len[b]
// goes to row t mod P of logical page t / P (physical page page_table[b][.])
// for every KV head, the page's summary absorbs the new key (it becomes the
// key itself when the token starts the page), then seq_len[b] = t + 1.  The
// summary stays the min/max over the page's written tokens, exactly as
// k_build_summaries would compute it.  A full sequence or an out-of-range
// page id sets KVR_ST_BAD_INDEX and leaves that sequence unchanged.
constexpr int kAppendThreads = 256;

template <int P>
__global__ void __launch_bounds__(kAppendThreads)
    k_append(const uint16_t *__restrict__ k_new, const uint16_t *__restrict__ v_new,
             const int32_t *__restrict__ page_table, int32_t *__restrict__ seq_len,
             uint16_t *__restrict__ k_pool, uint16_t *__restrict__ v_pool,
             uint16_t *__restrict__ summ, int H, int N, int n_phys) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int t = seq_len[b];  // read by every thread before the update below
  if (t < 0 || t >= N * P) {  // uniform over the CTA
    if (tid == 0) set_status(KVR_ST_BAD_INDEX);
    return;
  }
  const int p = t / P, r = t - p * P;
  const int phys = page_table[static_cast<size_t>(b) * N + p];
  if (phys < 0 || phys >= n_phys) {
    if (tid == 0) set_status(KVR_ST_BAD_INDEX);
    return;
  }
  // warp w takes heads w, w + 8, ...; lane l channels 4l .. 4l + 3
  for (int g = warp; g < H; g += kAppendThreads / 32) {
    const size_t src = (static_cast<size_t>(b) * H + g) * kD + 4 * lane;
    const uint2 kn = *reinterpret_cast<const uint2 *>(k_new + src);
    const uint2 vn = *reinterpret_cast<const uint2 *>(v_new + src);
    const size_t dst = ((static_cast<size_t>(phys) * P + r) * H + g) * kD + 4 * lane;
    *reinterpret_cast<uint2 *>(k_pool + dst) = kn;
    *reinterpret_cast<uint2 *>(v_pool + dst) = vn;
    uint16_t *sm = summ + ((static_cast<size_t>(b) * H + g) * N + p) * (2 * kD) + 4 * lane;
    uint2 mn = kn, mx = kn;
    if (r > 0) {
      const uint2 om = *reinterpret_cast<const uint2 *>(sm);
      const uint2 oM = *reinterpret_cast<const uint2 *>(sm + kD);
      const __nv_bfloat162 *a = reinterpret_cast<const __nv_bfloat162 *>(&om);
      const __nv_bfloat162 *c = reinterpret_cast<const __nv_bfloat162 *>(&oM);
      const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&kn);
      __nv_bfloat162 *m2 = reinterpret_cast<__nv_bfloat162 *>(&mn);
      __nv_bfloat162 *x2 = reinterpret_cast<__nv_bfloat162 *>(&mx);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        m2[i] = __hmin2(a[i], k2[i]);
        x2[i] = __hmax2(c[i], k2[i]);
      }
    }
    *reinterpret_cast<uint2 *>(sm) = mn;
    *reinterpret_cast<uint2 *>(sm + kD) = mx;
  }
  __syncthreads();
  if (tid == 0) seq_len[b] = t + 1;
}

}  // namespace kvr
