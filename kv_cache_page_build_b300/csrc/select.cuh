// select.cuh -- page scoring and top-k page selection per KV head, with the
// speculative mode's similarity test and correction.
//
// Sources: FreeKV (technical summary), section 1: KV retrieval keeps the
// whole cache and each step selects the part it needs; section 2.1: the
// selection is made per KV head, decisions are group-consistent (averaged
// over the group's query heads); speculative retrieval reuses the previous
// step's selection and fine-grained correction re-selects a KV head whose
// query similarity falls below tau.
//
// Score.  S[b][g][p] = (1/G) sum_{h in g} sum_c max(q_hc kmin_pc, q_hc kmax_pc).
// Because kmin <= kmax, max(q kmin, q kmax) is q kmax for q >= 0 and q kmin
// otherwise; with q+ = max(q, 0) and q- = min(q, 0) the term is
// fma(q+, kmax, fma(q-, kmin, .)) where one of the two products is an exact
// zero, so each channel adds exactly one exact bf16 x bf16 product to an fp32
// accumulator.  Every page is reduced in the same fixed order (channel pairs
// into two interleaved accumulators with packed FFMA2, the pair summed, G
// heads pairwise, then a 16-lane butterfly), so two pages with equal
// summaries get bitwise-equal scores.
//
// Layout of work.  Grid (splits, H, B): the N pages of a (b, g) row are cut
// into `splits` contiguous ranges, about two CTAs per SM in total.  A CTA's
// summaries are one contiguous byte range; its producer warp streams them
// with 1D bulk copies (32 pages = 16 KiB per copy) into a ring of stages,
// and the 8 consumer warps score every stage together (a half-warp per page,
// lane = 8 channels of the min and max rows).  Scores go to an fp32
// workspace row; the CTA that finishes the (b, g) row last (atomic ticket,
// no waiting) selects the top k.
//
// Top-k.  Scores map to order-preserving 32-bit keys (-0 folded into +0).
// The k-th largest key lies in a key interval [L, R], first [min, max].  A
// round cuts the interval into at most 2048 bins of 2^shift consecutive keys,
// histograms the keys inside it, and keeps the bin that holds the k-th
// largest (the keys of higher bins are selected).  Rounds repeat until the
// kept bin holds exactly as many keys as are still needed, or one key value
// only; among keys equal to that value the lowest page ids are taken (ties
// to the lower page id).  An ordered compaction writes the ids ascending.
#pragma once

#include "common.cuh"

namespace kvr {

constexpr int kSelConsumers = 8;                        // consumer warps
constexpr int kSelCT = 32 * kSelConsumers;              // consumer threads
constexpr int kSelThreads = kSelCT + 32;                // + one producer warp
constexpr int kSelStagePages = 32;                      // pages per bulk copy
constexpr int kSummBytes = 2 * kD * 2;                  // bytes of one page summary
constexpr int kSelStageBytes = kSelStagePages * kSummBytes;  // 16 KiB
constexpr int kSelStages = 6;
constexpr int kSelSmem = kSelStages * kSelStageBytes;   // 96 KiB: also holds N <= 16384 keys
constexpr int kSelBins = 2048;
static_assert(kSelSmem >= kMaxPages * 4, "the top-k keys reuse the stage ring");

struct SpecArgs {
  int enabled;                 // 0: plain selection
  int step;                    // 0 -> every head corrected
  float tau;                   // correction threshold
  uint16_t *q_prev;            // [B][Hq][D], read then replaced by q_t
  int32_t *sel_prev;           // [B][H][k], read then replaced by the new selection
  uint8_t *corrected;          // [B][H]
  float *cbar;                 // [B][H] or null
  int32_t *sel_used;           // [B][H][k]
  int32_t *sel_used_phys;      // [B][H][k] or null
  const int32_t *page2slot;    // [B][H][N] working-set map, or null (use page_table)
  int n_slots;                 // slots per sequence when page2slot is set
};

__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s + 0.0f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the kSelCT consumer threads (named barrier 1);
// `scratch` holds kSelConsumers words.  Also returns the total.
__device__ __forceinline__ uint32_t sel_exclusive_scan(uint32_t v, uint32_t *scratch,
                                                       uint32_t &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) scratch[warp] = incl;
  named_bar_sync(1, kSelCT);
  uint32_t base = 0u, tot = 0u;
#pragma unroll
  for (int w = 0; w < kSelConsumers; ++w) {
    const uint32_t x = scratch[w];
    base += w < warp ? x : 0u;
    tot += x;
  }
  total = tot;
  named_bar_sync(1, kSelCT);  // scratch free again
  return base + incl - v;
}

template <int G>
__global__ void __launch_bounds__(kSelThreads, (G <= 4 ? 2 : 1))
    k_score_select(const uint16_t *__restrict__ q, const uint16_t *__restrict__ summ,
                   const int32_t *__restrict__ page_table, int H, int N, int k, int n_split,
                   float *__restrict__ ws_scores, uint32_t *__restrict__ ws_count,
                   int32_t *__restrict__ sel_out, int32_t *__restrict__ sel_phys_out,
                   float *__restrict__ scores_out, SpecArgs spec) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kSelStages], empty[kSelStages];
  __shared__ uint32_t s_hist[kSelBins];
  __shared__ uint32_t s_scan[kSelConsumers];
  __shared__ uint32_t s_mm[2 * kSelConsumers];
  __shared__ uint32_t s_bin, s_bin_above, s_bin_cnt, s_last, s_corr;
  __shared__ float s_cos[8];
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int Hq = H * G;
  const size_t unit = static_cast<size_t>(b) * H + g;
  const int p0 = static_cast<int>(static_cast<long long>(split) * N / n_split);
  const int p1 = static_cast<int>(static_cast<long long>(split + 1) * N / n_split);
  const int np = p1 - p0;
  const int n_stages = (np + kSelStagePages - 1) / kSelStagePages;

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kSelStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSelConsumers);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ producer warp
  if (warp == kSelConsumers) {
    if (lane == 0) {
      const uint8_t *src = reinterpret_cast<const uint8_t *>(summ) + (unit * N + p0) * kSummBytes;
      int issued = 0;
      bool abort = false;
#pragma unroll 1
      for (int j = 0; j < n_stages; ++j) {
        const int s = j % kSelStages, use = j / kSelStages;
        if (use > 0 && !mbar_wait(&empty[s], static_cast<uint32_t>((use - 1) & 1))) abort = true;
        if (s_abort) abort = true;
        if (abort) {
          s_abort = 1;
          break;
        }
        const uint32_t bytes =
            static_cast<uint32_t>(min(kSelStagePages, np - j * kSelStagePages)) * kSummBytes;
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_copy_g2s(smem + s * kSelStageBytes,
                      src + static_cast<size_t>(j) * kSelStageBytes, bytes, &full[s]);
        issued = j + 1;
      }
      if (abort) {  // never leave with copies in flight
#pragma unroll 1
        for (int j = max(0, issued - kSelStages); j < issued; ++j)
          mbar_wait(&full[j % kSelStages], static_cast<uint32_t>((j / kSelStages) & 1));
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumer warps: scores
  const int ct = tid;
  {
    // this lane's query channels: 8 channels (8*sub .. 8*sub+7) of each head, as
    // sign-split pairs
    const int hw = ct >> 4, sub = ct & 15;
    float2 qp[G][4], qn[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(
          q + (static_cast<size_t>(b) * Hq + g * G + h) * kD + 8 * sub));
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 x = bf2_to_f2(w[j]);
        qp[h][j] = make_float2(fmaxf(x.x, 0.0f), fmaxf(x.y, 0.0f));
        qn[h][j] = make_float2(fminf(x.x, 0.0f), fminf(x.y, 0.0f));
      }
    }
    float *srow = ws_scores + unit * N + p0;
    float *orow = scores_out ? scores_out + unit * N + p0 : nullptr;
#pragma unroll 1
    for (int j = 0; j < n_stages; ++j) {
      const int s = j % kSelStages;
      bool have = false;
      if (__shfl_sync(0xffffffffu, s_abort, 0) == 0) {  // warp-uniform
        const bool ok = mbar_wait(&full[s], static_cast<uint32_t>((j / kSelStages) & 1));
        if (__all_sync(0xffffffffu, ok)) {
          have = true;
        } else if (lane == 0) {
          s_abort = 1;
        }
      }
      if (have) {
        const uint8_t *stage = smem + s * kSelStageBytes;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int pl = j * kSelStagePages + hw + 16 * r;  // page within this CTA's range
          const uint8_t *pg = stage + (hw + 16 * r) * kSummBytes;  // rows past np never written out
          const uint4 mn = *reinterpret_cast<const uint4 *>(pg + 16 * sub);
          const uint4 mx = *reinterpret_cast<const uint4 *>(pg + kD * 2 + 16 * sub);
          const uint32_t wn[4] = {mn.x, mn.y, mn.z, mn.w};
          const uint32_t wx[4] = {mx.x, mx.y, mx.z, mx.w};
          float2 acc2[G];
#pragma unroll
          for (int h = 0; h < G; ++h) acc2[h] = make_float2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float2 kmin = bf2_to_f2(wn[c]), kmax = bf2_to_f2(wx[c]);
#pragma unroll
            for (int h = 0; h < G; ++h) {
              acc2[h] = __ffma2_rn(qp[h][c], kmax, acc2[h]);
              acc2[h] = __ffma2_rn(qn[h][c], kmin, acc2[h]);
            }
          }
          float acc[G];
#pragma unroll
          for (int h = 0; h < G; ++h) acc[h] = acc2[h].x + acc2[h].y;
#pragma unroll
          for (int w = 1; w < G; w <<= 1)
#pragma unroll
            for (int h = 0; h < G; h += 2 * w) acc[h] += acc[h + w];
          float tot = acc[0];
#pragma unroll
          for (int m = 8; m >= 1; m >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, m);
          if (sub == 0 && pl < np) {
            const float sc = tot * (1.0f / G);
            srow[pl] = sc;
            if (orow) orow[pl] = sc;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }

  // ---- last CTA of this (b, g) row selects
  __threadfence();
  named_bar_sync(1, kSelCT);
  if (ct == 0) s_last = (atomicAdd(&ws_count[unit], 1u) == static_cast<uint32_t>(n_split - 1));
  named_bar_sync(1, kSelCT);
  if (!s_last) return;
  __threadfence();

  // keys of the whole row (the stage ring is idle now) and their range
  uint32_t *keys = reinterpret_cast<uint32_t *>(smem);
  uint32_t kmn = 0xffffffffu, kmx = 0u;
  for (int i = ct; i < N; i += kSelCT) {
    const uint32_t key = score_key(__ldcg(ws_scores + unit * N + i));
    keys[i] = key;
    kmn = min(kmn, key);
    kmx = max(kmx, key);
  }
  if (ct == 0) ws_count[unit] = 0u;  // leave the workspace zeroed
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    kmn = min(kmn, __shfl_xor_sync(0xffffffffu, kmn, m));
    kmx = max(kmx, __shfl_xor_sync(0xffffffffu, kmx, m));
  }
  if (lane == 0) {
    s_mm[warp] = kmn;
    s_mm[kSelConsumers + warp] = kmx;
  }
  named_bar_sync(1, kSelCT);
  uint32_t L = 0xffffffffu, R = 0u;
#pragma unroll
  for (int w = 0; w < kSelConsumers; ++w) {
    L = min(L, s_mm[w]);
    R = max(R, s_mm[kSelConsumers + w]);
  }
  // invariant: `need` of the `cnt` keys in [L, R] are still to be taken;
  // every key above R is taken
  uint32_t need = static_cast<uint32_t>(k), cnt = static_cast<uint32_t>(N);
#pragma unroll 1
  while (cnt != need && L != R) {
    const uint32_t span = R - L;
    const int shift = span < kSelBins ? 0 : (32 - __clz(span)) - 11;
    for (int i = ct; i < kSelBins; i += kSelCT) s_hist[i] = 0u;
    named_bar_sync(1, kSelCT);
    for (int i = ct; i < N; i += kSelCT) {
      const uint32_t key = keys[i];
      if (key >= L && key <= R) atomicAdd(&s_hist[(key - L) >> shift], 1u);
    }
    named_bar_sync(1, kSelCT);
    // thread ct owns bins [8 ct, 8 ct + 8); find the bin holding the need-th largest
    uint32_t c[kSelBins / kSelCT], mine = 0u;
#pragma unroll
    for (int e = 0; e < kSelBins / kSelCT; ++e) {
      c[e] = s_hist[(kSelBins / kSelCT) * ct + e];
      mine += c[e];
    }
    uint32_t total;
    const uint32_t below = sel_exclusive_scan(mine, s_scan, total);
    uint32_t above_here = total - below - mine;  // keys of the interval in higher bins
#pragma unroll
    for (int e = kSelBins / kSelCT - 1; e >= 0; --e) {
      if (above_here < need && need <= above_here + c[e]) {
        s_bin = static_cast<uint32_t>((kSelBins / kSelCT) * ct + e);
        s_bin_above = above_here;
        s_bin_cnt = c[e];
      }
      above_here += c[e];
    }
    named_bar_sync(1, kSelCT);
    const uint32_t nl = L + (s_bin << shift);
    const unsigned long long nr = static_cast<unsigned long long>(nl) + ((1ull << shift) - 1ull);
    need -= s_bin_above;
    cnt = s_bin_cnt;
    R = static_cast<uint32_t>(min(static_cast<unsigned long long>(R), nr));
    L = nl;
    named_bar_sync(1, kSelCT);  // s_bin* and s_hist free for the next round
  }

  // ---- speculative mode: group similarity and the correction decision
  const int32_t *ptab = page_table ? page_table + static_cast<size_t>(b) * N : nullptr;
  bool corrected = true;
  if (spec.enabled) {
    if (spec.step > 0 && warp < G) {
      const size_t base = (static_cast<size_t>(b) * Hq + g * G + warp) * kD + 4 * lane;
      const uint2 a = *reinterpret_cast<const uint2 *>(q + base);
      const uint2 c = *reinterpret_cast<const uint2 *>(spec.q_prev + base);
      const float x[4] = {bf_lo(a.x), bf_hi(a.x), bf_lo(a.y), bf_hi(a.y)};
      const float y[4] = {bf_lo(c.x), bf_hi(c.x), bf_lo(c.y), bf_hi(c.y)};
      float dot = 0.f, nx = 0.f, ny = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        dot = fmaf(x[i], y[i], dot);
        nx = fmaf(x[i], x[i], nx);
        ny = fmaf(y[i], y[i], ny);
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) {
        dot += __shfl_xor_sync(0xffffffffu, dot, m);
        nx += __shfl_xor_sync(0xffffffffu, nx, m);
        ny += __shfl_xor_sync(0xffffffffu, ny, m);
      }
      if (lane == 0) s_cos[warp] = (nx > 0.f && ny > 0.f) ? dot / (sqrtf(nx) * sqrtf(ny)) : 0.f;
    }
    named_bar_sync(1, kSelCT);
    if (ct == 0) {
      float cb = __int_as_float(0x7fc00000);  // NaN: no previous query at step 0
      bool corr = true;
      if (spec.step > 0) {
        float sum = 0.f;
        for (int h = 0; h < G; ++h) sum += s_cos[h];
        cb = sum / G;
        corr = cb < spec.tau;
      }
      s_corr = corr ? 1u : 0u;
      spec.corrected[unit] = corr ? 1 : 0;
      if (spec.cbar) spec.cbar[unit] = cb;
    }
    named_bar_sync(1, kSelCT);
    corrected = s_corr != 0u;
    // q_prev <- q_t for this group's heads (only this CTA reads them)
    for (int i = ct; i < G * kD / 8; i += kSelCT) {
      const size_t off = (static_cast<size_t>(b) * Hq + g * G) * kD + 8 * i;
      *reinterpret_cast<uint4 *>(spec.q_prev + off) = *reinterpret_cast<const uint4 *>(q + off);
    }
    if (!corrected) {  // reuse: sel_used <- previous selection (before it is replaced)
      for (int i = ct; i < k; i += kSelCT) {
        const int p = spec.sel_prev[unit * k + i];
        spec.sel_used[unit * k + i] = p;
        if (spec.sel_used_phys) {
          int phys = -1;
          if (p >= 0 && p < N)
            phys = spec.page2slot
                       ? (spec.page2slot[unit * N + p] >= 0
                              ? b * spec.n_slots + spec.page2slot[unit * N + p]
                              : -1)
                       : ptab[p];
          spec.sel_used_phys[unit * k + i] = phys;
        }
      }
    }
    named_bar_sync(1, kSelCT);
  }

  // ---- ordered compaction of the selection (ascending page ids): every key
  // above R, then the first `need` keys of [L, R] by page id (all of them
  // when cnt == need)
  const int per = (N + kSelCT - 1) / kSelCT;
  const int beg = min(N, ct * per), end = min(N, beg + per);
  uint32_t n_gt = 0u, n_eq = 0u;
  for (int i = beg; i < end; ++i) {
    const uint32_t key = keys[i];
    n_gt += (key > R);
    n_eq += (key >= L && key <= R);
  }
  uint32_t total;
  const uint32_t eq_base = sel_exclusive_scan(n_eq, s_scan, total);
  uint32_t n_take = n_gt;
  for (uint32_t e = 0; e < n_eq; ++e) n_take += (eq_base + e < need);
  uint32_t out = sel_exclusive_scan(n_take, s_scan, total);
  uint32_t eq_seen = 0u;
  for (int i = beg; i < end; ++i) {
    const uint32_t key = keys[i];
    bool take = key > R;
    if (key >= L && key <= R) take = (eq_base + eq_seen++) < need;
    if (!take) continue;
    if (out >= static_cast<uint32_t>(k)) break;  // never write past this unit's k entries
    const size_t o = unit * k + out++;
    if (spec.enabled) {
      spec.sel_prev[o] = i;
      if (corrected) {
        spec.sel_used[o] = i;
        if (spec.sel_used_phys && !spec.page2slot) spec.sel_used_phys[o] = ptab[i];
      }
    } else {
      sel_out[o] = i;
      if (sel_phys_out) sel_phys_out[o] = ptab[i];
    }
  }
}

}  // namespace kvr
