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
// Work decomposition.  The selected pages of all units form one flat list
// (unit-major, W = B * H * k pages; this is exactly the order of sel_phys).
// The grid is persistent: about one CTA per SM, CTA c owning the contiguous
// range [c W / n, (c + 1) W / n) of the list, so every CTA streams the same
// number of pages.  Where a range covers part of a unit, the CTA produces a
// partial (m, l, o) for that "segment"; the CTA that completes a unit's last
// segment (atomic ticket, no waiting) merges the unit's segments in segment
// order.  A unit whose pages all fall in one CTA is normalised directly.
//
// Inside a CTA.  Warp NC is the producer: its lanes fetch 32 page ids at a
// time and lane 0 issues, per page, one tiled TMA copy of the page's K rows
// and one of its V rows for head g (box D x 1 x P over the pool viewed as
// [tokens][H][D]) into a ring of S page stages (full/empty mbarriers per
// stage).  Warps 0..NC-1 (NC = 8, or 4 when fewer than 8 page stages fit)
// consume pages round-robin, one whole page per warp:
//   QK   LPT = 2G lanes per token, each holding 128/LPT channels of the G
//        query heads in registers (64 fp32 values for every G); products
//        are accumulated as fp32 pairs with packed FFMA2, and the G partial
//        dots are reduced over the LPT lanes by a transpose-reduction that
//        leaves head h in lanes 2h, 2h+1 of each token group.
//   softmax  online, base 2 (logits prescaled by scale * log2 e), per block
//        of up to 32 tokens: block max, rescale factor, p = 2^(x - m).
//   PV   lane = 4 channels of all G heads, p broadcast from shared memory as
//        (p, p) pairs, FFMA2 into the fp32 output accumulators.
// At the end of a segment the NC warps' states are combined in warp order.
// Every wait on a barrier is bounded; after a timeout the CTA stops
// issuing copies, drains the ones in flight, and still takes part in the
// tickets so the workspace counters stay consistent.
#pragma once

#include "common.cuh"

namespace kvr {

constexpr int kAttnMaxCtas = 1024;                         // bound on the persistent grid
constexpr int kAttnMinPagesPerCta = 4;
constexpr int kAttnSmemBytes = 227 * 1024 - 1024;          // dynamic shared memory budget

// Shared memory of the fixed (non-stage) areas for NC consumer warps.
template <int G>
constexpr int attn_fixed_bytes(int nc) {
  return nc * G * kD * 4      // combine area [NC][G][D] fp32
         + nc * G * 8         // combine (m, l) [NC][G]
         + nc * 32 * G * 8;   // p buffers [NC][32][G] (p, p)
}

template <int G, int P>
struct AttnCfg {
  static constexpr int kStageBytes = 2 * P * kD * 2;  // K and V of one page
  // 8 consumer warps when 8 stages fit, else 4: the ring needs S >= NC (see
  // the consumer's wait on the stage's previous use).
  static constexpr int NC =
      (kAttnSmemBytes - attn_fixed_bytes<G>(8)) / kStageBytes >= 8 ? 8 : 4;
  static constexpr int kThreads = 32 * (NC + 1);      // + one producer warp
  static constexpr int LPT = 2 * G;          // lanes per token in the QK pass
  static constexpr int TPI = 32 / LPT;       // tokens per QK iteration
  static constexpr int CH = 8 / G;           // 16-byte chunks of a K row per lane
  static constexpr int QP = 4 * CH;          // fp32 pairs of q per head per lane
  static constexpr int BT = P < 32 ? P : 32; // tokens per softmax block
  static constexpr int NBLK = P / BT;        // blocks per page
  static constexpr int IT = BT / TPI;        // QK iterations per block
  static constexpr int kCombBytes = NC * G * kD * 4;
  static constexpr int kCombMlBytes = NC * G * 8;
  static constexpr int kFixed = attn_fixed_bytes<G>(NC);
  static constexpr int kStagesFit = (kAttnSmemBytes - kFixed) / kStageBytes;
  static constexpr int S = kStagesFit > 24 ? 24 : kStagesFit;          // ring depth
  static constexpr int kSmem = S * kStageBytes + kFixed;
  static_assert(S >= NC, "the ring must have at least one stage per consumer warp");
  static_assert(IT * TPI == BT && NBLK * BT == P, "page tiling");
};

// Index of the CTA whose range holds flat page w (ranges start at c W / n).
__device__ __forceinline__ int attn_cta_of(long long w, long long W, int n) {
  return static_cast<int>(((w + 1) * n + W - 1) / W) - 1;
}

// Transpose-reduction of G values held by each of LPT lanes (sub = lane % LPT).
// On return the value is the full sum of head (sub >> 1).
template <int G, int LPT>
__device__ __forceinline__ float treduce(float (&v)[G], int sub) {
  int n = G;
#pragma unroll
  for (int m = LPT / 2; m >= 1; m >>= 1) {
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
      n = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
    }
  }
  return v[0];
}

__device__ __forceinline__ bool attn_unit_active(const uint8_t *filter, int filter_mode,
                                                 long long u) {
  if (filter_mode == 0) return true;
  return (filter[u] != 0) == (filter_mode == 2);
}

// filter_mode: 0 every unit; 1 only units with filter[unit] == 0; 2 only != 0
template <int G, int P>
__global__ void __launch_bounds__(AttnCfg<G, P>::kThreads, 1)
    k_sparse_decode(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const uint16_t *__restrict__ q,
                    const int32_t *__restrict__ sel_phys, int H, int k, int n_phys, long long W,
                    float scale_log2, const uint8_t *__restrict__ filter, int filter_mode,
                    float *__restrict__ part_o, float2 *__restrict__ part_ml,
                    uint32_t *__restrict__ counters, float *__restrict__ out) {
  using C = AttnCfg<G, P>;
  constexpr int S = C::S;
  constexpr int NC = C::NC;
  extern __shared__ __align__(128) uint8_t smem[];
  float *comb_o = reinterpret_cast<float *>(smem + S * C::kStageBytes);
  float2 *comb_ml = reinterpret_cast<float2 *>(smem + S * C::kStageBytes + C::kCombBytes);
  float2 *pbuf_all =
      reinterpret_cast<float2 *>(smem + S * C::kStageBytes + C::kCombBytes + C::kCombMlBytes);
  __shared__ __align__(8) uint64_t full[S], empty[S];
  __shared__ int s_ok[S];
  __shared__ volatile int s_abort;
  __shared__ uint32_t s_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_ctas = gridDim.x, cta = blockIdx.x;
  const long long w0 = cta * W / n_ctas, w1 = (cta + 1) * W / n_ctas;

  if (tid == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
#pragma unroll 1
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ producer warp
  if (warp == NC) {
    int issued = 0;  // local pages issued so far
    bool abort = false;
#pragma unroll 1
    for (long long base = w0; base < w1 && !abort; base += 32) {
      const int n = static_cast<int>(min(32LL, w1 - base));
      int id = -1, g = 0, act = 0;
      if (lane < n) {
        const long long w = base + lane;
        const long long u = w / k;
        id = __ldg(sel_phys + w);
        g = static_cast<int>(u % H);
        act = attn_unit_active(filter, filter_mode, u) ? 1 : 0;
      }
#pragma unroll 1
      for (int j = 0; j < n; ++j) {
        const int pid = __shfl_sync(0xffffffffu, id, j);
        const int pg = __shfl_sync(0xffffffffu, g, j);
        const int pact = __shfl_sync(0xffffffffu, act, j);
        if (lane == 0 && !abort) {
          const int i = static_cast<int>(base + j - w0);
          const int s = i % S;
          const int use = i / S;
          if (use > 0 && !mbar_wait(&empty[s], static_cast<uint32_t>((use - 1) & 1))) abort = true;
          if (s_abort) abort = true;
          if (abort) {
            s_abort = 1;
          } else {
            const bool ok = pact && pid >= 0 && pid < n_phys;
            s_ok[s] = ok ? 1 : 0;
            if (ok) {
              uint8_t *dst = smem + s * C::kStageBytes;
              mbar_arrive_expect_tx(&full[s], C::kStageBytes);
              tma_load_3d(dst, &tmap_k, &full[s], 0, pg, pid * P);
              tma_load_3d(dst + P * kD * 2, &tmap_v, &full[s], 0, pg, pid * P);
            } else {
              if (pact) set_status(KVR_ST_BAD_INDEX);
              mbar_arrive(&full[s]);
            }
            issued = i + 1;
          }
        }
      }
      abort = __shfl_sync(0xffffffffu, abort ? 1 : 0, 0) != 0;
    }
    if (lane == 0 && abort) {  // never leave with copies in flight
#pragma unroll 1
      for (int i = max(0, issued - S); i < issued; ++i)
        mbar_wait(&full[i % S], static_cast<uint32_t>((i / S) & 1));
    }
    return;
  }

  // ------------------------------------------------------------ consumer warps
  using Cfg = C;
  const int cw = warp;
  const int sub = lane % Cfg::LPT, grp = lane / Cfg::LPT, hd = sub >> 1;
  const int ct = tid;  // 0 .. 32 * NC - 1
  constexpr int kCT = 32 * NC;
  float2 *pbuf = pbuf_all + cw * 32 * G;
  const int Hq = H * G;
  const long long u_first = w0 / k, u_last = (w1 - 1) / k;

#pragma unroll 1
  for (long long u = u_first; u <= u_last; ++u) {
    const long long seg_lo = max(w0, u * k), seg_hi = min(w1, (u + 1) * k);
    const bool active = attn_unit_active(filter, filter_mode, u);
    const int b = static_cast<int>(u / H), g = static_cast<int>(u % H);

    // this lane's q channels: chunks sub + LPT*j (8 channels each) of every head
    float2 q2[G][Cfg::QP];
    if (active) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const uint16_t *qh = q + (static_cast<size_t>(b) * Hq + g * G + h) * kD;
#pragma unroll
        for (int j = 0; j < Cfg::CH; ++j) {
          const uint4 w = __ldg(reinterpret_cast<const uint4 *>(qh + 8 * (sub + Cfg::LPT * j)));
          q2[h][4 * j + 0] = bf2_to_f2(w.x);
          q2[h][4 * j + 1] = bf2_to_f2(w.y);
          q2[h][4 * j + 2] = bf2_to_f2(w.z);
          q2[h][4 * j + 3] = bf2_to_f2(w.w);
        }
      }
    }
    float m_run = -INFINITY, l_run = 0.f;
    float2 o2[G][2];
#pragma unroll
    for (int h = 0; h < G; ++h) o2[h][0] = o2[h][1] = make_float2(0.f, 0.f);

    const int i_lo = static_cast<int>(seg_lo - w0), i_hi = static_cast<int>(seg_hi - w0);
    int i = i_lo + (cw - i_lo % NC + NC) % NC;
#pragma unroll 1
    for (; i < i_hi; i += NC) {
      const int s = i % S, use = i / S;
      bool have = false;
      if (__shfl_sync(0xffffffffu, s_abort, 0) == 0) {  // warp-uniform
        // Pages go to the warps round-robin, so this warp can reach use `use`
        // of stage s before use - 1 (another warp's page) has landed; a
        // parity wait on `full` alone would then see use - 1's phase.  Wait
        // first until use - 1 is released: by then every page up to
        // i - NC - S has been consumed (the producer issued this warp's
        // previous page i - NC), so with S >= NC both parity waits below are
        // unambiguous.
        bool ok = use == 0 || mbar_wait(&empty[s], static_cast<uint32_t>((use - 1) & 1));
        if (ok) ok = mbar_wait(&full[s], static_cast<uint32_t>(use & 1));
        if (__all_sync(0xffffffffu, ok)) {
          have = s_ok[s] != 0;
        } else if (lane == 0) {
          s_abort = 1;
        }
      }
      if (have && active) {
        const uint16_t *sk = reinterpret_cast<const uint16_t *>(smem + s * C::kStageBytes);
        const uint16_t *sv = sk + P * kD;
#pragma unroll 1
        for (int blk = 0; blk < Cfg::NBLK; ++blk) {
          const uint16_t *kb = sk + blk * Cfg::BT * kD;
          const uint16_t *vb = sv + blk * Cfg::BT * kD;
          // ---- QK
          float xs[Cfg::IT];
#pragma unroll
          for (int it = 0; it < Cfg::IT; ++it) {
            const uint16_t *row = kb + (it * Cfg::TPI + grp) * kD;
            float2 acc2[G];
#pragma unroll
            for (int h = 0; h < G; ++h) acc2[h] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < Cfg::CH; ++j) {
              const uint4 w = *reinterpret_cast<const uint4 *>(row + 8 * (sub + Cfg::LPT * j));
              const float2 k0 = bf2_to_f2(w.x), k1 = bf2_to_f2(w.y);
              const float2 k2 = bf2_to_f2(w.z), k3 = bf2_to_f2(w.w);
#pragma unroll
              for (int h = 0; h < G; ++h) {
                acc2[h] = __ffma2_rn(q2[h][4 * j + 0], k0, acc2[h]);
                acc2[h] = __ffma2_rn(q2[h][4 * j + 1], k1, acc2[h]);
                acc2[h] = __ffma2_rn(q2[h][4 * j + 2], k2, acc2[h]);
                acc2[h] = __ffma2_rn(q2[h][4 * j + 3], k3, acc2[h]);
              }
            }
            float acc[G];
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] = acc2[h].x + acc2[h].y;
            xs[it] = treduce<G, Cfg::LPT>(acc, sub) * scale_log2;
          }
          // ---- online softmax for this block (head hd in this lane)
          float bm = xs[0];
#pragma unroll
          for (int it = 1; it < Cfg::IT; ++it) bm = fmaxf(bm, xs[it]);
#pragma unroll
          for (int m = Cfg::LPT; m < 32; m <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, m));
          const float m_new = fmaxf(m_run, bm);
          const float alpha = exp2f(m_run - m_new);
          float ps = 0.f;
#pragma unroll
          for (int it = 0; it < Cfg::IT; ++it) {
            const float p = exp2f(xs[it] - m_new);
            ps += p;
            if ((sub & 1) == 0) pbuf[(it * Cfg::TPI + grp) * G + hd] = make_float2(p, p);
          }
#pragma unroll
          for (int m = Cfg::LPT; m < 32; m <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, m);
          l_run = fmaf(l_run, alpha, ps);
          m_run = m_new;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float a = __shfl_sync(0xffffffffu, alpha, 2 * h);
            const float2 a2 = make_float2(a, a);
            o2[h][0] = __fmul2_rn(o2[h][0], a2);
            o2[h][1] = __fmul2_rn(o2[h][1], a2);
          }
          __syncwarp();
          // ---- PV
#pragma unroll 4
          for (int t = 0; t < Cfg::BT; ++t) {
            const uint2 vw = *reinterpret_cast<const uint2 *>(vb + t * kD + 4 * lane);
            const float2 v0 = bf2_to_f2(vw.x), v1 = bf2_to_f2(vw.y);
            if constexpr (G == 1) {
              const float2 p = pbuf[t];
              o2[0][0] = __ffma2_rn(p, v0, o2[0][0]);
              o2[0][1] = __ffma2_rn(p, v1, o2[0][1]);
            } else {
#pragma unroll
              for (int h = 0; h < G; h += 2) {
                const float4 pp = *reinterpret_cast<const float4 *>(pbuf + t * G + h);
                const float2 pa = make_float2(pp.x, pp.y), pb = make_float2(pp.z, pp.w);
                o2[h][0] = __ffma2_rn(pa, v0, o2[h][0]);
                o2[h][1] = __ffma2_rn(pa, v1, o2[h][1]);
                o2[h + 1][0] = __ffma2_rn(pb, v0, o2[h + 1][0]);
                o2[h + 1][1] = __ffma2_rn(pb, v1, o2[h + 1][1]);
              }
            }
          }
          __syncwarp();
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!active) continue;  // uniform over the consumer warps

    // ---- combine the 8 warps' states of this segment (warp order)
    if (grp == 0 && (sub & 1) == 0) comb_ml[cw * G + hd] = make_float2(m_run, l_run);
#pragma unroll
    for (int h = 0; h < G; ++h)
      *reinterpret_cast<float4 *>(comb_o + (cw * G + h) * kD + 4 * lane) =
          make_float4(o2[h][0].x, o2[h][0].y, o2[h][1].x, o2[h][1].y);
    named_bar_sync(1, kCT);

    const int c_first = attn_cta_of(u * k, W, n_ctas);
    const int n_segs = attn_cta_of((u + 1) * k - 1, W, n_ctas) - c_first + 1;
    const size_t slot = static_cast<size_t>(cta) + static_cast<size_t>(u);
    float *orow = out + (static_cast<size_t>(b) * Hq + g * G) * kD;
#pragma unroll 1
    for (int e = ct; e < G * kD; e += kCT) {
      const int h = e / kD, ch = e - h * kD;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NC; ++w) M = fmaxf(M, comb_ml[w * G + h].x);
      float L = 0.f, A = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NC; ++w) {
          const float2 ml = comb_ml[w * G + h];
          const float sc = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
          L = fmaf(sc, ml.y, L);
          A = fmaf(sc, comb_o[(w * G + h) * kD + ch], A);
        }
      }
      if (n_segs == 1) {
        if (L <= 0.f && ch == 0) set_status(KVR_ST_NO_TOKENS);
        orow[e] = L > 0.f ? A / L : 0.f;
      } else {
        part_o[slot * G * kD + e] = A;
        if (ch == 0) part_ml[slot * G + h] = make_float2(M, L);
      }
    }
    if (n_segs > 1) {
      __threadfence();
      named_bar_sync(1, kCT);
      if (ct == 0) s_last = (atomicAdd(&counters[u], 1u) == static_cast<uint32_t>(n_segs - 1));
      named_bar_sync(1, kCT);
      if (s_last) {
        __threadfence();
        // merge the unit's segments in segment (CTA) order
#pragma unroll 1
        for (int e = ct; e < G * kD; e += kCT) {
          const int h = e / kD, ch = e - h * kD;
          float M = -INFINITY;
#pragma unroll 1
          for (int j = 0; j < n_segs; ++j)
            M = fmaxf(M, __ldcg(part_ml + (static_cast<size_t>(c_first + j) + u) * G + h).x);
          float L = 0.f, A = 0.f;
          if (M != -INFINITY) {
#pragma unroll 4
            for (int j = 0; j < n_segs; ++j) {
              const size_t sl = static_cast<size_t>(c_first + j) + static_cast<size_t>(u);
              const float2 ml = __ldcg(part_ml + sl * G + h);
              const float sc = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
              L = fmaf(sc, ml.y, L);
              A = fmaf(sc, __ldcg(part_o + sl * G * kD + e), A);
            }
          }
          if (L <= 0.f && ch == 0) set_status(KVR_ST_NO_TOKENS);
          orow[e] = L > 0.f ? A / L : 0.f;
        }
        if (ct == 0) counters[u] = 0u;
      }
    }
    named_bar_sync(1, kCT);  // comb buffers free for the next segment
  }
}

}  // namespace kvr
