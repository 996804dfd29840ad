// attention.cuh -- split-K GQA decode attention over the selected pages.
//
// Source: FreeKV (technical summary), section 2.1: the attention of a decode
// step runs on the retrieved KV pages only; "Key-Value (KV) Cache" wiki page:
// decode attention is bound by memory bandwidth; grouped-query attention.
//
// For sequence b and KV head g (a "unit"), the G query heads of the group
// attend over the tokens of the unit's k selected pages:
//   out[b][h] = sum_t softmax_t(scale * q_h . K_t) V_t .
//
// Layout of work.  Grid (splits, H, B); a CTA (128 threads, 4 warps) takes
// 128 consecutive tokens of the unit's selection (128 / P pages).  Its thread
// 0 issues one tiled TMA copy per page for K and one for V (box D x 1 x P over
// the pool viewed as [tokens][H][D]: one head's P rows, 256 bytes each), all
// up front, each on its own mbarrier, so the CTA's whole 64 KiB is in flight
// at once.  Then, from shared memory:
//   QK: 8 lanes per token, each lane 16 channels (two 16-byte reads: one in
//       each half of the row, conflict-free) of the G heads; the G partial
//       dot products are reduced over the 8 lanes by a transpose-reduction
//       (halving the value set at each step), leaving head h in lanes 2h, 2h+1.
//   softmax: one warp per head, base-2 exponentials of logits prescaled by
//       scale * log2(e); the CTA keeps (m, l) per head.
//   PV: each warp takes 32 consecutive tokens; lane = 4 channels of all G
//       heads; the 4 warps' partial outputs are summed in a fixed order.
// Each CTA writes (m, l, o) per head; the CTA that finishes its unit last
// (atomic ticket, no waiting) rescales and sums the splits in split order and
// writes the fp32 output.  A unit with one split normalises directly.
#pragma once

#include "common.cuh"

namespace kvr {

constexpr int kAttnThreads = 128;
constexpr int kAttnTokens = 128;                        // tokens per CTA
constexpr int kAttnTileBytes = kAttnTokens * kD * 2;    // 32 KiB of K (same for V)

__host__ __device__ constexpr int attn_pages_per_cta(int P) { return kAttnTokens / P; }

__host__ __device__ inline int attn_splits(int k, int P) {
  const int ppc = kAttnTokens / P;
  return (k + ppc - 1) / ppc;
}

// Transpose-reduction of G values held by each of 8 lanes (sub = lane & 7).
// On return v[0] holds the full sum of head `head` in this lane.
template <int G>
__device__ __forceinline__ float reduce8(float (&v)[G], int sub, int &head) {
  int n = G;
  head = 0;
#pragma unroll
  for (int m = 4; m >= 1; m >>= 1) {
    if (n > 1) {
      const bool up = (sub & m) != 0;
      const int half = n / 2;
#pragma unroll
      for (int i = 0; i < G / 2; ++i) {
        if (i < half) {
          const float send = up ? v[i] : v[i + half];
          const float keep = up ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
      }
      if (up) head += half;
      n = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
    }
  }
  return v[0];
}

// filter_mode: 0 every unit; 1 only units with filter[unit] == 0; 2 only != 0
template <int G, int P>
__global__ void __launch_bounds__(kAttnThreads)
    k_sparse_decode(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const uint16_t *__restrict__ q,
                    const int32_t *__restrict__ sel_phys, int H, int k, int n_phys,
                    int n_splits, float scale_log2, const uint8_t *__restrict__ filter,
                    int filter_mode, float *__restrict__ part_o, float *__restrict__ part_ml,
                    uint32_t *__restrict__ counters, float *__restrict__ out) {
  constexpr int PPC = kAttnTokens / P;
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t *sk = reinterpret_cast<uint16_t *>(smem);                   // [128][D]
  uint16_t *sv = reinterpret_cast<uint16_t *>(smem + kAttnTileBytes);  // [128][D]
  float *s_p = reinterpret_cast<float *>(smem + 2 * kAttnTileBytes);  // [128][G]
  __shared__ __align__(8) uint64_t bar_k[PPC], bar_v[PPC];
  __shared__ int s_valid[PPC];
  __shared__ float s_m[G], s_l[G];
  __shared__ uint32_t s_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int Hq = H * G;
  const size_t unit = static_cast<size_t>(b) * H + g;
  if (filter_mode != 0) {
    const bool corr = filter[unit] != 0;
    if ((filter_mode == 1) == corr) return;  // the whole unit belongs to the other launch
  }
  const int page0 = split * PPC;
  const int npages = min(PPC, k - page0);
  const int ntok = npages * P;

  if (tid == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    for (int i = 0; i < PPC; ++i) {
      mbar_init(&bar_k[i], 1);
      mbar_init(&bar_v[i], 1);
    }
    fence_barrier_init();
    for (int i = 0; i < npages; ++i) {
      const int phys = sel_phys[unit * k + page0 + i];
      const bool ok = phys >= 0 && phys < n_phys;
      s_valid[i] = ok;
      if (!ok) {
        set_status(KVR_ST_BAD_INDEX);
        continue;
      }
      mbar_arrive_expect_tx(&bar_k[i], P * kD * 2);
      tma_load_3d(sk + i * P * kD, &tmap_k, &bar_k[i], 0, g, phys * P);
    }
    for (int i = 0; i < npages; ++i) {
      if (!s_valid[i]) continue;
      const int phys = sel_phys[unit * k + page0 + i];
      mbar_arrive_expect_tx(&bar_v[i], P * kD * 2);
      tma_load_3d(sv + i * P * kD, &tmap_v, &bar_v[i], 0, g, phys * P);
    }
  }

  // query registers: this lane's 16 channels (8*sub.. and 64+8*sub..) of each head
  const int sub = lane & 7, grp = lane >> 3;
  float qr[G][16];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint16_t *qh = q + (static_cast<size_t>(b) * Hq + g * G + h) * kD;
    unpack8(*reinterpret_cast<const uint4 *>(qh + 8 * sub), &qr[h][0]);
    unpack8(*reinterpret_cast<const uint4 *>(qh + 64 + 8 * sub), &qr[h][8]);
  }
  __syncthreads();

  // ---- QK: warp w, step it handles token it*16 + w*4 + grp
  bool timed_out = false;
  int waited = -1;
#pragma unroll 1
  for (int it = 0; it * 16 < ntok; ++it) {
    const int t = it * 16 + warp * 4 + grp;
    const int pg = min(t, ntok - 1) / P;
    const int pg_hi = min(it * 16 + warp * 4 + 3, ntok - 1) / P;  // warp-uniform wait range
    for (int w = waited + 1; w <= pg_hi; ++w)
      if (s_valid[w] && !mbar_wait(&bar_k[w], 0)) timed_out = true;
    waited = max(waited, pg_hi);
    const uint16_t *row = sk + t * kD;
    float kf[16];
    unpack8(*reinterpret_cast<const uint4 *>(row + 8 * sub), &kf[0]);
    unpack8(*reinterpret_cast<const uint4 *>(row + 64 + 8 * sub), &kf[8]);
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float a = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) a = fmaf(qr[h][c], kf[c], a);
      acc[h] = a;
    }
    int head;
    const float dot = reduce8<G>(acc, sub, head);
    const int writer_mask = (G >= 8) ? 0 : (G == 4 ? 1 : (G == 2 ? 3 : 7));
    if ((sub & writer_mask) == 0 && t < ntok)
      s_p[t * G + head] = s_valid[pg] ? dot * scale_log2 : -INFINITY;
  }
  __syncthreads();

  // ---- softmax statistics per head (base 2)
  for (int h = warp; h < G; h += kAttnThreads / 32) {
    float m = -INFINITY;
    for (int t = lane; t < ntok; t += 32) m = fmaxf(m, s_p[t * G + h]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
    for (int t = lane; t < kAttnTokens; t += 32) {
      float p = 0.f;
      if (t < ntok && m != -INFINITY) p = exp2f(s_p[t * G + h] - m);
      s_p[t * G + h] = p;
      l += p;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) {
      s_m[h] = m;
      s_l[h] = l;
    }
  }
  __syncthreads();

  // ---- PV: warp w takes tokens [32w, 32w + 32); lane = channels 4*lane .. +3
  float o[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[h][c] = 0.f;
  {
    const int t_beg = warp * 32, t_end = min(ntok, t_beg + 32);
    int cur = -1;
#pragma unroll 4
    for (int t = t_beg; t < t_end; ++t) {
      const int pg = t / P;
      if (pg != cur) {
        cur = pg;
        if (s_valid[pg] && !mbar_wait(&bar_v[pg], 0)) timed_out = true;
      }
      if (!s_valid[pg]) continue;
      const uint2 raw = *reinterpret_cast<const uint2 *>(sv + t * kD + 4 * lane);
      const float v[4] = {bf_lo(raw.x), bf_hi(raw.x), bf_lo(raw.y), bf_hi(raw.y)};
      float p[G];
#pragma unroll
      for (int h = 0; h < G; ++h) p[h] = s_p[t * G + h];
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[h][c] = fmaf(p[h], v[c], o[h][c]);
    }
  }
  if (timed_out) {  // never leave with copies in flight
    for (int i = 0; i < npages; ++i)
      if (s_valid[i]) {
        mbar_wait(&bar_k[i], 0);
        mbar_wait(&bar_v[i], 0);
      }
  }
  __syncthreads();  // K/V tiles no longer read: reuse the K area for the warp sums

  float *red = reinterpret_cast<float *>(smem);  // [4][G][D]
#pragma unroll
  for (int h = 0; h < G; ++h)
    *reinterpret_cast<float4 *>(red + (warp * G + h) * kD + 4 * lane) =
        make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
  __syncthreads();

  if (n_splits == 1) {  // the only split: normalise and write the output
    for (int i = tid; i < G * kD; i += kAttnThreads) {
      const int h = i / kD, c = i - h * kD;
      const float s = ((red[(0 * G + h) * kD + c] + red[(1 * G + h) * kD + c]) +
                       red[(2 * G + h) * kD + c]) + red[(3 * G + h) * kD + c];
      const float l = s_l[h];
      if (l <= 0.f && c == 0) set_status(KVR_ST_NO_TOKENS);
      out[(static_cast<size_t>(b) * Hq + g * G + h) * kD + c] = l > 0.f ? s / l : 0.f;
    }
    return;
  }

  const size_t part = unit * n_splits + split;
  for (int i = tid; i < G * kD; i += kAttnThreads) {
    const int h = i / kD, c = i - h * kD;
    part_o[(part * G + h) * kD + c] = ((red[(0 * G + h) * kD + c] + red[(1 * G + h) * kD + c]) +
                                       red[(2 * G + h) * kD + c]) + red[(3 * G + h) * kD + c];
  }
  if (tid < G) {
    part_ml[(part * G + tid) * 2 + 0] = s_m[tid];
    part_ml[(part * G + tid) * 2 + 1] = s_l[tid];
  }

  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&counters[unit], 1u) == static_cast<uint32_t>(n_splits - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- merge the unit's splits in split order
  const float *pm = part_ml + unit * n_splits * G * 2;
  const float *po = part_o + unit * n_splits * G * kD;
  for (int i = tid; i < G * kD; i += kAttnThreads) {
    const int h = i / kD, c = i - h * kD;
    float M = -INFINITY;
    for (int s = 0; s < n_splits; ++s) M = fmaxf(M, __ldcg(pm + (s * G + h) * 2));
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll 4
      for (int s = 0; s < n_splits; ++s) {
        const float ms = __ldcg(pm + (s * G + h) * 2);
        const float w = ms == -INFINITY ? 0.f : exp2f(ms - M);
        L = fmaf(w, __ldcg(pm + (s * G + h) * 2 + 1), L);
        acc = fmaf(w, __ldcg(po + (s * G + h) * kD + c), acc);
      }
    }
    if (L <= 0.f && c == 0) set_status(KVR_ST_NO_TOKENS);
    out[(static_cast<size_t>(b) * Hq + g * G + h) * kD + c] = L > 0.f ? acc / L : 0.f;
  }
  if (tid == 0) counters[unit] = 0u;
}

}  // namespace kvr
