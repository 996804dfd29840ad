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

template <int P>
__global__ void __launch_bounds__(kSumThreads)
    k_build_summaries(const uint16_t *__restrict__ k_pool, const int32_t *__restrict__ page_table,
                      uint16_t *__restrict__ summ, int H, int N, int n_phys, int pages_per_cta) {
  const int cols = H * 16;  // 16-byte columns per token row
  const int b = blockIdx.y;
  const size_t token_stride = static_cast<size_t>(H) * kD;  // elements between tokens
  for (int idx = threadIdx.x; idx < pages_per_cta * cols; idx += kSumThreads) {
    const int pl = idx / cols;
    const int col = idx - pl * cols;
    const int p = blockIdx.x * pages_per_cta + pl;
    if (p >= N) continue;
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
          } else {
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

}  // namespace kvr
