// recall.cuh -- streamed recall of selected pages from a host-resident cache.
//
// Source: FreeKV (technical summary), section 2.2: the host copy of the cache
// is head-major (HND) so that a page of one head is one contiguous transfer,
// the GPU copy is token-major (NHD) so that decode needs no transposes, and
// the layout changes only when pages move between the two; recall is
// double-buffered so transfer and conversion overlap the computation.
//
// One CTA per (sequence b, KV head g):
//   plan   - slots holding a page of the new selection or of the protected
//            selection (the one the running attention reads) are kept; the
//            new selection's non-resident pages (ascending page id) take the
//            free slots (ascending slot id); both maps are updated.
//   gather - the CTA copies each missed page's P x D block of K and of V from
//            page-locked host memory (loads through the host mapping, 16
//            bytes per lane, eight loads in flight per lane) into the slot's
//            token-major stripe of head g: the HND -> NHD conversion happens
//            in the same pass as the transfer.
// With n_slots >= 2k the two sets of k pages always fit: one set is read by
// the running step while the other is being filled.
//
// unit_filter splits one recall into two launches over disjoint units (the
// units never share a slot, a map entry or a page): 0 = every unit, 1 = the
// units with corrected == 0 (the speculative prefetch for the next step),
// 2 = the units with corrected != 0 (the pages this step still needs).
#pragma once

#include "common.cuh"

namespace kvr {

constexpr int kRecallThreads = 256;

// Ordered compaction helper: each thread owns a contiguous range of `n`
// candidates; returns the output position of its first kept candidate.
template <typename Pred>
__device__ __forceinline__ uint32_t ordered_base(int n, Pred keep, uint32_t *scratch,
                                                 uint32_t &total, int &beg, int &end) {
  const int per = (n + kRecallThreads - 1) / kRecallThreads;
  beg = min(n, static_cast<int>(threadIdx.x) * per);
  end = min(n, beg + per);
  uint32_t cnt = 0;
  for (int i = beg; i < end; ++i) cnt += keep(i) ? 1u : 0u;
  return block_exclusive_scan<kRecallThreads>(cnt, scratch, total);
}

template <int P>
__global__ void __launch_bounds__(kRecallThreads)
    k_recall(const uint16_t *__restrict__ k_host, const uint16_t *__restrict__ v_host,
             uint16_t *__restrict__ k_slots, uint16_t *__restrict__ v_slots,
             int32_t *__restrict__ page2slot, int32_t *__restrict__ slot2page, int S,
             const int32_t *__restrict__ sel_new, const int32_t *__restrict__ protect,
             const uint8_t *__restrict__ corrected, int unit_filter, int H, int N, int k,
             int32_t *__restrict__ sel_slot_out, uint32_t *__restrict__ n_copied) {
  extern __shared__ __align__(16) int32_t rsm[];
  int32_t *keep = rsm;               // [S]
  int32_t *free_list = rsm + S;      // [S]
  int32_t *miss = rsm + 2 * S;       // [k]
  __shared__ uint32_t s_scan[kRecallThreads / 32];

  const int tid = threadIdx.x;
  const int g = blockIdx.x, b = blockIdx.y;
  const size_t unit = static_cast<size_t>(b) * H + g;
  if (unit_filter != 0 && corrected != nullptr &&
      (unit_filter == 2) != (corrected[unit] != 0))
    return;  // the whole CTA leaves before its first barrier
  int32_t *p2s = page2slot + unit * N;
  int32_t *s2p = slot2page + unit * S;
  const int32_t *sn = sel_new + unit * k;
  const int32_t *pr = protect + unit * k;

  for (int s = tid; s < S; s += kRecallThreads) keep[s] = 0;
  __syncthreads();
  for (int i = tid; i < k; i += kRecallThreads) {
    const int a = sn[i], c = pr[i];
    if (a >= 0 && a < N && p2s[a] >= 0 && p2s[a] < S) keep[p2s[a]] = 1;
    if (c >= 0 && c < N && p2s[c] >= 0 && p2s[c] < S) keep[p2s[c]] = 1;
  }
  __syncthreads();

  // misses of the new selection, in selection (ascending page) order
  auto is_miss = [&](int i) { const int a = sn[i]; return a >= 0 && a < N && p2s[a] < 0; };
  uint32_t n_miss, n_free;
  int beg, end;
  uint32_t pos = ordered_base(k, is_miss, s_scan, n_miss, beg, end);
  for (int i = beg; i < end; ++i)
    if (is_miss(i)) miss[pos++] = sn[i];
  auto is_free = [&](int s) { return keep[s] == 0; };
  pos = ordered_base(S, is_free, s_scan, n_free, beg, end);
  for (int s = beg; s < end; ++s)
    if (is_free(s)) free_list[pos++] = s;
  __syncthreads();
  if (n_miss > n_free) {
    if (tid == 0) set_status(KVR_ST_NO_FREE_SLOT);
    n_miss = n_free;
  }

  // update the maps (evicted pages and missed pages are distinct entries)
  for (int i = tid; i < static_cast<int>(n_miss); i += kRecallThreads) {
    const int s = free_list[i], p = miss[i];
    const int old = s2p[s];
    if (old >= 0 && old < N) p2s[old] = -1;
    p2s[p] = s;
    s2p[s] = p;
  }

  // gather: job = (miss i, K or V, token t, 16-byte column j)
  const int per_page = 2 * P * 16;
  const int jobs = static_cast<int>(n_miss) * per_page;
  const size_t stripe = static_cast<size_t>(H) * kD;  // slot elements between tokens
  constexpr int U = 8;
  for (int base = tid; base < jobs; base += U * kRecallThreads) {
    uint4 v[U];
    uint16_t *dst[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int idx = base + u * kRecallThreads;
      dst[u] = nullptr;
      if (idx < jobs) {
        const int i = idx / per_page;
        const int r = idx - i * per_page;
        const int kv = r / (P * 16);
        const int t = (r / 16) % P;
        const int j = r & 15;
        const int p = miss[i], s = free_list[i];
        const uint16_t *src = (kv ? v_host : k_host) + ((unit * N + p) * P + t) * kD + 8 * j;
        v[u] = *reinterpret_cast<const uint4 *>(src);
        dst[u] = (kv ? v_slots : k_slots) +
                 ((static_cast<size_t>(b) * S + s) * P + t) * stripe + static_cast<size_t>(g) * kD +
                 8 * j;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (dst[u]) *reinterpret_cast<uint4 *>(dst[u]) = v[u];
  }
  __syncthreads();

  if (corrected && corrected[unit]) {
    for (int i = tid; i < k; i += kRecallThreads) {
      const int p = pr[i];
      const int s = (p >= 0 && p < N) ? p2s[p] : -1;
      sel_slot_out[unit * k + i] = s >= 0 ? b * S + s : -1;
    }
  }
  if (tid == 0 && n_copied && n_miss) atomicAdd(n_copied, n_miss);
}

}  // namespace kvr
