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
// Work decomposition.  The selected pages of all units, cut into chunks of
// C = min(P, 32) tokens, form one flat list (unit-major, the order of
// sel_phys).  Every consumer warp of the grid is an independent "worker":
// worker v of n owns the contiguous range [v W / n, (v + 1) W / n) of the
// list, so all workers stream the same number of chunks.  Where a range
// covers part of a unit, the worker writes a partial (m, l, o) for that
// "segment" straight from its registers; k_attn_merge, launched right after,
// merges each split unit's segments in segment order.  A unit whose chunks
// all fall in one worker's range is normalised directly.
//
// Inside a CTA (CPS per SM, all resident) the warps share nothing but the
// shared-memory ring:
//   producer  warp NC; lane w feeds consumer warp w, which owns R stages of
//        the ring: as soon as the warp releases a stage, the lane issues the
//        warp's next chunk into it (four tiled TMA copies: the 64-channel
//        halves of the chunk's K and V rows for head g, 128-byte swizzled).
//        The range's page ids are read into shared memory first, so issuing
//        never waits on a load.
//   consumer  warps 0..NC-1 on the tensor cores (mma.sync m16n8k16, bf16 in,
//        fp32 accumulators):
//     QK   S[h][t] = q_h . K_t, the G query heads on the 16-row side (rows
//          G..15 zero), 8 tokens per MMA column block; q stays in registers
//          as A fragments, K fragments come from shared memory by ldmatrix.
//     softmax  online, base 2 (logits prescaled by scale * log2 e), per
//          chunk, on the accumulator fragments (4 lanes per head).
//     PV   O^T[c][h] += V^T[c][t] P^T[t][h]: V fragments by transposing
//          ldmatrix, P straight from the QK accumulators, split into a bf16
//          high part and a bf16 residual (two MMAs) so the weights keep
//          about 16 bits.
// The G x D output of a group is a 4- to 32-row contraction per page, far
// from the tensor cores' peak; they are used because they cut the issue
// slots per chunk about five-fold against CUDA-core FMAs, which keeps the
// consumers well ahead of the memory stream.
// Every wait is bounded; after a timeout the CTA stops issuing copies and
// drains the ones in flight.
#pragma once

#include "common.cuh"

namespace kvr {

constexpr int kAttnNC = 3;                         // consumer warps per CTA
constexpr int kAttnThreads = 32 * (kAttnNC + 1);   // + one producer warp
constexpr int kAttnMaxCtas = 512;                  // bound on the grid
constexpr int kAttnMaxWorkers = kAttnMaxCtas * kAttnNC;
constexpr int kAttnMinChunksPerWorker = 2;
constexpr int kAttnIds = 128;                      // page ids of a worker range kept in shared memory
constexpr int kAttnCPS = 2;                        // CTAs per SM
constexpr int kSmemPerSM = 228 * 1024;             // shared memory of one SM

template <int G, int P>
struct AttnCfg {
  static constexpr int C = P < 32 ? P : 32;        // tokens per chunk (one stage)
  static constexpr int CPP = P / C;                // chunks per page
  static constexpr int NB = C / 8;                 // 8-token column blocks of the QK MMA
  static constexpr int KP = C / 16;                // 16-token k-steps of the PV MMA
  static constexpr int kHalf = C * 128;            // 64 channels of C rows (swizzled)
  static constexpr int kStageBytes = 4 * kHalf;    // K lo, K hi, V lo, V hi
  static constexpr int R = 32768 / kStageBytes;    // stages per consumer warp (32 KiB)
  static constexpr int S = kAttnNC * R;            // ring depth
  static constexpr int kSmem = S * kStageBytes + 1024;  // + 1 KiB to align the ring
  static_assert(kAttnCPS * (kSmem + 2048 + 4 * kAttnNC * kAttnIds) <= kSmemPerSM,
                "CTAs per SM must fit");
  static_assert(CPP * C == P && NB * 8 == C && KP * 16 == C && R >= 2, "chunk tiling");
};

// Index of the worker (or CTA) whose range holds flat chunk w (ranges start
// at c W / n).
__device__ __forceinline__ int attn_cta_of(long long w, long long W, int n) {
  return static_cast<int>(((w + 1) * n + W - 1) / W) - 1;
}

__device__ __forceinline__ bool attn_unit_active(const uint8_t *filter, int filter_mode,
                                                 long long u) {
  if (filter_mode == 0) return true;
  return (filter[u] != 0) == (filter_mode == 2);
}

// One chunk of C tokens for head row gq of a consumer warp: QK on the tensor
// cores, online-softmax update of (m_run, l_run) and O^T += V^T P^T.
template <int G, int P>
__device__ __forceinline__ void attn_chunk(uint32_t kb, const uint32_t (&qa)[8][2],
                                           float scale_log2, float &m_run, float &l_run,
                                           float (&o)[8][4], int lane) {
  using Cfg = AttnCfg<G, P>;
  constexpr int HALF = Cfg::kHalf;
  const int gq = lane >> 2, tq = lane & 3, mi = lane >> 3, mr = lane & 7;
  const uint32_t vb = kb + 2 * HALF;
  // ---- QK: sc[nb] = S[gq][8 nb + 2 tq (+1)]
  float sc[Cfg::NB][4];
#pragma unroll
  for (int nb = 0; nb < Cfg::NB; ++nb) {
    sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
#pragma unroll
    for (int kq = 0; kq < 4; ++kq) {  // channel chunks 4kq .. 4kq+3 = k-steps 2kq, 2kq+1
      uint32_t bf[4];
      ldsm_x4(swz<HALF>(kb, 8 * nb + mr, 4 * kq + mi), bf);
      mma_bf16_16816(sc[nb], qa[2 * kq][0], 0u, qa[2 * kq][1], 0u, bf[0], bf[1]);
      mma_bf16_16816(sc[nb], qa[2 * kq + 1][0], 0u, qa[2 * kq + 1][1], 0u, bf[2], bf[3]);
    }
  }
  // ---- online softmax for head gq (4 lanes per head, 2 tokens per block each)
  float mx = -INFINITY;
#pragma unroll
  for (int nb = 0; nb < Cfg::NB; ++nb) {
    sc[nb][0] *= scale_log2;
    sc[nb][1] *= scale_log2;
    mx = fmaxf(mx, fmaxf(sc[nb][0], sc[nb][1]));
  }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const float m_new = fmaxf(m_run, mx);
  const float alpha = exp2f(m_run - m_new);
  const bool row_on = gq < G;
  float ls = 0.f;
#pragma unroll
  for (int nb = 0; nb < Cfg::NB; ++nb) {
    const float p0 = row_on ? exp2f(sc[nb][0] - m_new) : 0.f;
    const float p1 = row_on ? exp2f(sc[nb][1] - m_new) : 0.f;
    sc[nb][0] = p0;
    sc[nb][1] = p1;
    ls += p0 + p1;
  }
  l_run = fmaf(l_run, alpha, ls);
  m_run = m_new;
  // rescale O: this lane's columns are heads 2tq and 2tq + 1
  const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * tq);
  const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * tq + 4);
#pragma unroll
  for (int mb = 0; mb < 8; ++mb) {
    o[mb][0] *= a0;
    o[mb][1] *= a1;
    o[mb][2] *= a0;
    o[mb][3] *= a1;
  }
  // ---- P^T as B fragments: high bf16 part and bf16 residual
  uint32_t ph[Cfg::KP][2], pl[Cfg::KP][2];
#pragma unroll
  for (int kp = 0; kp < Cfg::KP; ++kp)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float x0 = sc[2 * kp + e][0], x1 = sc[2 * kp + e][1];
      const uint32_t hi = pack_bf16x2(x0, x1);
      ph[kp][e] = hi;
      pl[kp][e] = pack_bf16x2(x0 - __uint_as_float(hi << 16),
                              x1 - __uint_as_float(hi & 0xffff0000u));
    }
  // ---- PV: O^T[16 mb ..][heads] += V^T[16 mb ..][16 kp ..] P^T
#pragma unroll
  for (int mb = 0; mb < 8; ++mb) {
#pragma unroll
    for (int kp = 0; kp < Cfg::KP; ++kp) {
      uint32_t va[4];
      ldsm_x4_trans(swz<HALF>(vb, 16 * kp + 8 * (mi >> 1) + mr, 2 * mb + (mi & 1)), va);
      mma_bf16_16816(o[mb], va[0], va[1], va[2], va[3], ph[kp][0], ph[kp][1]);
      mma_bf16_16816(o[mb], va[0], va[1], va[2], va[3], pl[kp][0], pl[kp][1]);
    }
  }
}

// filter_mode: 0 every unit; 1 only units with filter[unit] == 0; 2 only != 0
template <int G, int P>
__global__ void __launch_bounds__(kAttnThreads, kAttnCPS)
    k_sparse_decode(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const uint16_t *__restrict__ q,
                    const int32_t *__restrict__ sel_phys, int H, int k, int n_phys, long long W,
                    float scale_log2, const uint8_t *__restrict__ filter, int filter_mode,
                    float *__restrict__ part_o, float2 *__restrict__ part_ml,
                    float *__restrict__ out) {
  using Cfg = AttnCfg<G, P>;
  constexpr int NC = kAttnNC, CPP = Cfg::CPP, HALF = Cfg::kHalf, R = Cfg::R, S = Cfg::S;
  extern __shared__ uint8_t smem_raw[];
  // the swizzle pattern repeats every 1024 bytes: align the ring to it
  uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  const uint32_t ring = smem_addr(smem);
  __shared__ __align__(8) uint64_t full[S], empty[S];
  __shared__ int s_ok[S];
  __shared__ int s_ids[NC][kAttnIds];  // page ids of the first kAttnIds chunks of each worker
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_workers = gridDim.x * NC;
  const long long kc = static_cast<long long>(k) * CPP;  // chunks per unit

  if (tid == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
#pragma unroll
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // Launched as a programmatic dependent launch, this kernel's setup above
  // overlaps the previous kernel; every global read and write comes after
  // this wait.  Then the merge kernel may be scheduled.
  pdl_wait();
  if (tid == 0) pdl_launch_dependents();

  // ------------------------------------------------------------ producer warp
  if (warp == NC) {
    // page ids of the workers' ranges, once, so that issuing never waits on a load
#pragma unroll 1
    for (int w = 0; w < NC; ++w) {
      const long long v = static_cast<long long>(blockIdx.x) * NC + w;
      const long long a = v * W / n_workers, n = (v + 1) * W / n_workers - a;
      for (int j = lane; j < n && j < kAttnIds; j += 32) s_ids[w][j] = __ldg(sel_phys + (a + j) / CPP);
    }
    __syncwarp();
    // lane w (< NC) feeds consumer warp w: the worker's chunks go to its R
    // stages in turn.  The lane walks them incrementally: unit u, chunk
    // position pos in the unit, KV head g = u % H.
    const bool feeder = lane < NC;
    const long long v = static_cast<long long>(blockIdx.x) * NC + lane;
    const long long a = v * W / n_workers;
    const int n = feeder ? static_cast<int>((v + 1) * W / n_workers - a) : 0;
    int i = 0;
    long long u = a / kc, pos = a % kc;
    int g = static_cast<int>(u % H);
    bool abort = false;
    uint64_t t_prog = global_timer_ns();
#pragma unroll 1
    while (true) {
      const bool mine = i < n && !abort;
      if (!__any_sync(0xffffffffu, mine)) break;
      if (mine) {
        const int s = lane * R + i % R;
        if (i < R || mbar_test_wait(&empty[s], static_cast<uint32_t>((i / R - 1) & 1))) {
          const int id = i < kAttnIds ? s_ids[lane][i] : __ldg(sel_phys + u * k + pos / CPP);
          const bool act = attn_unit_active(filter, filter_mode, u);
          const bool ok = act && id >= 0 && id < n_phys;
          s_ok[s] = ok ? 1 : 0;
          if (ok) {
            uint8_t *dst = smem + s * Cfg::kStageBytes;
            const int row = id * P + static_cast<int>(pos % CPP) * Cfg::C;
            mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
            tma_load_3d(dst, &tmap_k, &full[s], 0, g, row);
            tma_load_3d(dst + HALF, &tmap_k, &full[s], 64, g, row);
            tma_load_3d(dst + 2 * HALF, &tmap_v, &full[s], 0, g, row);
            tma_load_3d(dst + 3 * HALF, &tmap_v, &full[s], 64, g, row);
          } else {
            if (act) set_status(KVR_ST_BAD_INDEX);
            mbar_arrive(&full[s]);
          }
          ++i;
          if (++pos == kc) {
            pos = 0;
            ++u;
            g = g + 1 == H ? 0 : g + 1;
          }
          t_prog = global_timer_ns();
        } else if (global_timer_ns() - t_prog > kWaitNs) {
          set_status(KVR_ST_WAIT_TIMEOUT);
          s_abort = 1;
        }
        if (s_abort) abort = true;
      }
    }
    // never leave with copies in flight: after an abort, wait (bounded) for
    // this lane's last issued chunks
    if (feeder && abort)
      for (int j = max(0, i - R); j < i; ++j)
        mbar_wait(&full[lane * R + j % R], static_cast<uint32_t>((j / R) & 1));
    return;
  }

  // ------------------------------------------------------------ consumer warps
  const int cw = warp;
  const int gq = lane >> 2, tq = lane & 3;  // MMA fragment row group and column pair
  const int Hq = H * G;
  const long long v = static_cast<long long>(blockIdx.x) * NC + cw;  // this worker
  const long long a = v * W / n_workers;
  const int n = static_cast<int>((v + 1) * W / n_workers - a);

  uint32_t qa[8][2];            // q of head gq as A fragments (k-step kk: channels 16kk + 2tq, +8)
  float m_run, l_run;           // per head gq; l_run is this lane's partial
  float o[8][4];                // O^T[16 mb + gq (+8)][2 tq (+1)]
  long long u = a / kc, pos = a % kc;

  // Close the segment of unit `uu`: a partial for a split unit, the
  // normalised output for a unit that lies in this range alone.
  auto flush = [&](long long uu) {
    if (!attn_unit_active(filter, filter_mode, uu)) return;  // uniform over the warp
    float l = l_run;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const int c_first = attn_cta_of(uu * kc, W, n_workers);
    const int n_segs = attn_cta_of((uu + 1) * kc - 1, W, n_workers) - c_first + 1;
    if (n_segs == 1) {
      const int b = static_cast<int>(uu / H), g = static_cast<int>(uu % H);
      float *orow = out + (static_cast<size_t>(b) * Hq + g * G) * kD;
      const float la = __shfl_sync(0xffffffffu, l, 8 * tq);      // head 2tq
      const float lb = __shfl_sync(0xffffffffu, l, 8 * tq + 4);  // head 2tq + 1
      if (tq == 0 && gq < G && l <= 0.f) set_status(KVR_ST_NO_TOKENS);
#pragma unroll
      for (int mb = 0; mb < 8; ++mb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int head = 2 * tq + (e & 1), ch = 16 * mb + gq + 8 * (e >> 1);
          const float lh = (e & 1) ? lb : la;
          if (head < G) orow[head * kD + ch] = lh > 0.f ? o[mb][e] / lh : 0.f;
        }
    } else {
      const size_t slot = static_cast<size_t>(v) + static_cast<size_t>(uu);
      float *po = part_o + slot * G * kD;
      if (tq == 0 && gq < G) part_ml[slot * G + gq] = make_float2(m_run, l);
#pragma unroll
      for (int mb = 0; mb < 8; ++mb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int head = 2 * tq + (e & 1), ch = 16 * mb + gq + 8 * (e >> 1);
          if (head < G) po[head * kD + ch] = o[mb][e];
        }
    }
  };
  auto start = [&](long long uu) {  // new segment: zero state, q of the unit
    m_run = -INFINITY;
    l_run = 0.f;
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) o[mb][0] = o[mb][1] = o[mb][2] = o[mb][3] = 0.f;
    const int b = static_cast<int>(uu / H), g = static_cast<int>(uu % H);
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
        q + (static_cast<size_t>(b) * Hq + g * G + min(gq, G - 1)) * kD);
    const bool on = gq < G;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qa[kk][0] = on ? __ldg(qrow + 8 * kk + tq) : 0u;
      qa[kk][1] = on ? __ldg(qrow + 8 * kk + 4 + tq) : 0u;
    }
  };

  start(u);
#pragma unroll 1
  for (int i = 0; i < n; ++i) {
    if (i > 0 && pos == 0) {  // the range enters the next unit
      flush(u - 1);
      start(u);
    }
    const int s = cw * R + i % R;  // this warp's stages in turn
    bool have = false;
    if (__shfl_sync(0xffffffffu, s_abort, 0) == 0) {  // warp-uniform
      const bool ok = mbar_wait(&full[s], static_cast<uint32_t>((i / R) & 1));
      if (__all_sync(0xffffffffu, ok)) {
        have = s_ok[s] != 0;
      } else if (lane == 0) {
        s_abort = 1;
      }
    }
    if (have) attn_chunk<G, P>(ring + s * Cfg::kStageBytes, qa, scale_log2, m_run, l_run, o, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (++pos == kc) {
      pos = 0;
      ++u;
    }
  }
  if (n > 0) flush(pos == 0 ? u - 1 : u);
}

// Merge of the split units, launched right after k_sparse_decode on the same
// stream as a programmatic dependent launch (its CTAs may be scheduled while
// k_sparse_decode runs; pdl_wait holds them until it has completed and its
// partials are visible).  One CTA per (unit, query head of the group), one
// thread per channel: the thread folds the unit's segments in segment order,
// kMG at a time with all of their loads in flight, rescaling online.
constexpr int kMG = 16;

template <int G>
__global__ void __launch_bounds__(kD)
    k_attn_merge(const float *__restrict__ part_o, const float2 *__restrict__ part_ml, int H,
                 long long kc, long long W, int n_workers, const uint8_t *__restrict__ filter,
                 int filter_mode, float *__restrict__ out) {
  // every CTA waits, so this kernel never completes before k_sparse_decode
  // (later work on the stream may rewrite what k_sparse_decode reads)
  pdl_wait();
  const long long u = blockIdx.x / G;
  const int h = blockIdx.x % G, ch = threadIdx.x;
  const int c_first = attn_cta_of(u * kc, W, n_workers);
  const int n_segs = attn_cta_of((u + 1) * kc - 1, W, n_workers) - c_first + 1;
  if (n_segs == 1 || !attn_unit_active(filter, filter_mode, u)) return;  // written by the main kernel
  const size_t slot0 = static_cast<size_t>(c_first) + static_cast<size_t>(u);
  float M = -INFINITY, L = 0.f, A = 0.f;
#pragma unroll 1
  for (int j0 = 0; j0 < n_segs; j0 += kMG) {
    float2 ml[kMG];
    float ov[kMG];
#pragma unroll
    for (int j = 0; j < kMG; ++j) {
      const size_t sl = slot0 + min(j0 + j, n_segs - 1);
      ml[j] = __ldg(part_ml + sl * G + h);
      ov[j] = __ldg(part_o + (sl * G + h) * kD + ch);
    }
    // no early exits below: every load above is consumed in straight-line
    // code, so the compiler keeps them all in flight together
    float bm = M;
#pragma unroll
    for (int j = 0; j < kMG; ++j) bm = fmaxf(bm, j0 + j < n_segs ? ml[j].x : -INFINITY);
    const float rs = M == -INFINITY ? 0.f : exp2f(M - bm);
    L *= rs;
    A *= rs;
#pragma unroll
    for (int j = 0; j < kMG; ++j) {
      const bool on = j0 + j < n_segs && ml[j].x != -INFINITY;
      const float sc = on ? exp2f(ml[j].x - bm) : 0.f;
      L = fmaf(sc, ml[j].y, L);
      A = fmaf(sc, ov[j], A);
    }
    M = bm;
  }
  const int b = static_cast<int>(u / H), g = static_cast<int>(u % H);
  if (L <= 0.f && ch == 0) set_status(KVR_ST_NO_TOKENS);
  out[((static_cast<size_t>(b) * H + g) * G + h) * kD + ch] = L > 0.f ? A / L : 0.f;
}

}  // namespace kvr
