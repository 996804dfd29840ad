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
// accumulator.  Every page is reduced in the same fixed order (8 channels
// per lane in order, G heads pairwise, then a 16-lane butterfly), so two
// pages with equal summaries get bitwise-equal scores.
//
// Layout of work.  Grid (chunks, H, B).  A CTA scores 64 consecutive pages of
// one (b, g): it pulls their 64 x 512-byte summaries into shared memory with
// four 8 KiB bulk copies (one mbarrier each) and a half-warp scores one page
// at a time (lane = 8 channels, 16-byte shared loads of the min and max
// rows).  Scores go to an fp32 workspace row; the CTA that finishes the
// (b, g) row last (atomic ticket, no waiting) selects the top k.
//
// Top-k.  Scores map to order-preserving 32-bit keys (-0 folded into +0).  A
// most-significant-digit radix select (8-bit digits, shared-memory
// histograms) finds the k-th largest key; pages above it are selected, and
// among pages equal to it the lowest ids fill the remaining places (ties to
// the lower page id).  An ordered compaction writes the ids ascending.
#pragma once

#include "common.cuh"

namespace kvr {

constexpr int kSelThreads = 256;
constexpr int kSelChunk = 64;                   // pages per scoring CTA
constexpr int kSummBytes = 2 * kD * 2;          // bytes of one page summary
constexpr int kSelStageBytes = kSelChunk * kSummBytes;  // 32 KiB
static_assert(kSelThreads == 256, "one histogram bin per thread");

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

template <int G>
__global__ void __launch_bounds__(kSelThreads)
    k_score_select(const uint16_t *__restrict__ q, const uint16_t *__restrict__ summ,
                   const int32_t *__restrict__ page_table, int H, int N, int k, int n_chunks,
                   float *__restrict__ ws_scores, uint32_t *__restrict__ ws_count,
                   int32_t *__restrict__ sel_out, int32_t *__restrict__ sel_phys_out,
                   float *__restrict__ scores_out, SpecArgs spec) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[4];
  __shared__ uint32_t s_hist[256];
  __shared__ uint32_t s_scan[kSelThreads / 32];
  __shared__ uint32_t s_prefix, s_mask, s_need, s_done, s_last, s_corr;
  __shared__ float s_cos[8];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.y, b = blockIdx.z;
  const int Hq = H * G;
  const size_t unit = static_cast<size_t>(b) * H + g;
  const int p0 = blockIdx.x * kSelChunk;
  const int np = min(kSelChunk, N - p0);

  // ---- stage the chunk's summaries (4 bulk copies of up to 16 pages)
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
    const uint8_t *src = reinterpret_cast<const uint8_t *>(summ) + (unit * N + p0) * kSummBytes;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int cnt = min(16, np - 16 * i);
      if (cnt > 0) {
        const uint32_t bytes = static_cast<uint32_t>(cnt) * kSummBytes;
        mbar_arrive_expect_tx(&bars[i], bytes);
        bulk_copy_g2s(smem + i * 16 * kSummBytes, src + i * 16 * kSummBytes, bytes, &bars[i]);
      }
    }
  }

  // ---- this lane's query channels: 8 channels (8*sub .. 8*sub+7) of each head
  const int hw = tid >> 4, sub = tid & 15;
  float qp[G][8], qn[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint4 raw = *reinterpret_cast<const uint4 *>(
        q + (static_cast<size_t>(b) * Hq + g * G + h) * kD + 8 * sub);
    float x[8];
    unpack8(raw, x);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      qp[h][c] = fmaxf(x[c], 0.0f);
      qn[h][c] = fminf(x[c], 0.0f);
    }
  }
  __syncthreads();  // barrier initialisation visible to all threads

  // ---- score: half-warp hw takes page 16*i + hw of the chunk
  bool timed_out = false;
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    if (16 * i >= np) break;  // uniform over the CTA
    if (!mbar_wait(&bars[i], 0)) timed_out = true;
    const int pl = 16 * i + hw;
    const uint8_t *pg = smem + pl * kSummBytes;  // rows beyond np are never written out
    float kmin[8], kmax[8];
    unpack8(*reinterpret_cast<const uint4 *>(pg + 16 * sub), kmin);
    unpack8(*reinterpret_cast<const uint4 *>(pg + kD * 2 + 16 * sub), kmax);
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float a = 0.0f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        a = fmaf(qp[h][c], kmax[c], a);
        a = fmaf(qn[h][c], kmin[c], a);
      }
      acc[h] = a;
    }
#pragma unroll
    for (int w = 1; w < G; w <<= 1)
#pragma unroll
      for (int h = 0; h < G; h += 2 * w) acc[h] += acc[h + w];
    float tot = acc[0];
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, m);
    if (sub == 0 && pl < np) ws_scores[unit * N + p0 + pl] = tot * (1.0f / G);
  }
  if (timed_out) {  // never leave the CTA with copies in flight
    for (int i = 0; i < 4; ++i)
      if (16 * i < np) mbar_wait(&bars[i], 0);
  }

  // ---- last CTA of this (b, g) row selects
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&ws_count[unit], 1u) == static_cast<uint32_t>(n_chunks - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  uint32_t *keys = reinterpret_cast<uint32_t *>(smem);  // the staging area is free now
  for (int i = tid; i < N; i += kSelThreads) {
    const float s = __ldcg(ws_scores + unit * N + i);
    keys[i] = score_key(s);
    if (scores_out) scores_out[unit * N + i] = s;
  }
  if (tid == 0) ws_count[unit] = 0u;  // leave the workspace zeroed
  __syncthreads();

  // radix select of the k-th largest key: prefix/mask = digits fixed so far,
  // need = how many of the keys matching the prefix still have to be taken
  uint32_t prefix = 0u, mask = 0u, need = static_cast<uint32_t>(k);
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    s_hist[tid] = 0u;  // kSelThreads == 256 bins
    __syncthreads();
    for (int i = tid; i < N; i += kSelThreads) {
      const uint32_t key = keys[i];
      if ((key & mask) == prefix) atomicAdd(&s_hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t c[8], sum = 0u;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = s_hist[255 - 8 * lane - i];  // lane 0 holds the highest digits
        sum += c[i];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - sum;
      if (excl < need && need <= incl) {
        uint32_t above = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (above + c[i] >= need) {
            const uint32_t digit = static_cast<uint32_t>(255 - 8 * lane - i);
            s_prefix = prefix | (digit << shift);
            s_mask = mask | (255u << shift);
            s_need = need - above;
            s_done = (c[i] == need - above) ? 1u : 0u;
            break;
          }
          above += c[i];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    mask = s_mask;
    need = s_need;
    if (s_done) break;  // every key with this prefix is taken
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
    __syncthreads();
    if (tid == 0) {
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
    __syncthreads();
    corrected = s_corr != 0u;
    // q_prev <- q_t for this group's heads (only this CTA reads them)
    for (int i = tid; i < G * kD / 8; i += kSelThreads) {
      const size_t off = (static_cast<size_t>(b) * Hq + g * G) * kD + 8 * i;
      *reinterpret_cast<uint4 *>(spec.q_prev + off) = *reinterpret_cast<const uint4 *>(q + off);
    }
    if (!corrected) {  // reuse: sel_used <- previous selection (before it is replaced)
      for (int i = tid; i < k; i += kSelThreads) {
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
    __syncthreads();
  }

  // ---- ordered compaction of the selection (ascending page ids)
  const int per = (N + kSelThreads - 1) / kSelThreads;
  const int beg = min(N, tid * per), end = min(N, beg + per);
  uint32_t n_gt = 0u, n_eq = 0u;
  for (int i = beg; i < end; ++i) {
    const uint32_t m = keys[i] & mask;
    n_gt += (m > prefix);
    n_eq += (m == prefix);
  }
  uint32_t total;
  const uint32_t eq_base = block_exclusive_scan<kSelThreads>(n_eq, s_scan, total);
  uint32_t n_take = n_gt;
  for (uint32_t e = 0; e < n_eq; ++e) n_take += (eq_base + e < need);
  uint32_t out = block_exclusive_scan<kSelThreads>(n_take, s_scan, total);
  uint32_t eq_seen = 0u;
  for (int i = beg; i < end; ++i) {
    const uint32_t m = keys[i] & mask;
    bool take = m > prefix;
    if (m == prefix) take = (eq_base + eq_seen++) < need;
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
