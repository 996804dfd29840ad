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
// zero, so each channel adds exactly one exact bf16 x bf16 product.  Per unit
// this is a contraction [q- | q+] (G x 256) . [kmin ; kmax] (256 x pages):
// it runs on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 out) with the
// pages on the 16-row side and the G heads as columns, then the G head scores
// of a page are summed in a fixed order (in-lane pair, then an xor butterfly
// over the column pairs).  Two pages with equal summaries go through
// identical operations, so they get bitwise-equal scores.
//
// Two kernels.
//   k_page_scores streams the summaries.  The rows of all (b, g) units form
//   one flat list of 512-byte page summaries, viewed by TMA as [pages][256];
//   every consumer warp of the grid is an independent worker over a
//   contiguous range of it.  Its producer lane loads the range 32 pages
//   (16 KiB: four 64-channel boxes, 128-byte swizzled) at a time, never
//   across a unit boundary (a shorter stage takes 8-page boxes), into the
//   worker's R private stages; the worker scores a stage with 32 MMAs fed by
//   ldmatrix.
//   k_topk, one CTA per unit, launched right after as a programmatic
//   dependent launch, reads the unit's N scores and selects.
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

constexpr int kSummBytes = 2 * kD * 2;                     // bytes of one page summary
constexpr int kScNC = 3;                                   // workers (consumer warps) per CTA
constexpr int kScThreads = 32 * (kScNC + 1);               // + one producer warp
constexpr int kScPages = 32;                               // pages per stage
constexpr int kScStageBytes = kScPages * kSummBytes;       // 16 KiB
constexpr int kScR = 2;                                    // stages per worker
constexpr int kScS = kScNC * kScR;
constexpr int kScCPS = 2;                                  // CTAs per SM
constexpr int kScSmem = kScS * kScStageBytes + 1024;       // 96 KiB + alignment of the ring
constexpr int kScMaxCtas = 512;
constexpr int kScMinPagesPerWorker = 32;
constexpr int kSelBins = 2048;

struct SpecArgs {
  int enabled;                 // 0: plain selection
  int decided;                 // 1: k_spec_decide has already taken the decision and
                               //    filled sel_used for the reused heads; the top-k
                               //    only reads `corrected` and writes the selections
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
  unsigned long long *ready;   // [B][H] or null: a reused unit's word is set to ready_tag
                               //    (release) once its sel_used and sel_used_phys are
                               //    written, so the attention may start it early
  unsigned long long ready_tag;
};

__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s + 0.0f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Next stage of a worker: from flat page f (page pos of its unit), at most 32
// pages, never past the unit's end or the range end e.
// v F / n (a worker's range boundary in the flat page list) and f = u N + pos,
// with 32-bit division whenever the operands fit (64-bit division is emulated
// and would sit on the path to the first copy).
__device__ __forceinline__ long long flat_split(long long v, long long F, int n) {
  const unsigned long long p = static_cast<unsigned long long>(v) * static_cast<unsigned long long>(F);
  if (p <= 0xffffffffull) return static_cast<long long>(static_cast<uint32_t>(p) / static_cast<uint32_t>(n));
  return static_cast<long long>(p / static_cast<unsigned long long>(n));
}
__device__ __forceinline__ void flat_divmod(long long f, int N, long long &u, int &pos) {
  if (f <= 0xffffffffll) {
    const uint32_t q = static_cast<uint32_t>(f) / static_cast<uint32_t>(N);
    u = q;
    pos = static_cast<int>(static_cast<uint32_t>(f) - q * static_cast<uint32_t>(N));
  } else {
    u = f / N;
    pos = static_cast<int>(f - u * N);
  }
}

__device__ __forceinline__ int sc_chunk(long long f, int pos, int N, long long e) {
  return static_cast<int>(min(static_cast<long long>(min(kScPages, N - pos)), e - f));
}

// NR query rows per unit: the G heads of the group times the T query tokens
// of the step (q [B][T][Hq][D]); the score is the mean over the NR rows.
// Rows take the MMA's 8 columns, in CB blocks.
template <int NR>
__global__ void __launch_bounds__(kScThreads, kScCPS)
    k_page_scores(const __grid_constant__ CUtensorMap tmap_s, const __grid_constant__ CUtensorMap tmap_s8,
                  const uint16_t *__restrict__ q, int H, int N, long long F, int T, int G,
                  uint64_t wait_ns, float *__restrict__ ws_scores, float *__restrict__ scores_out) {
  constexpr int CB = NR > 8 ? 2 : 1;
  constexpr int HALF = kScPages * 128;  // one 64-channel box of a stage
  extern __shared__ uint8_t smem_raw[];
  // the swizzle pattern repeats every 1024 bytes: align the ring to it
  uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  const uint32_t ring = smem_addr(smem);
  __shared__ __align__(8) uint64_t full[kScS], empty[kScS];
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_workers = gridDim.x * kScNC;
  const int Hq = H * G;

  if (tid == 0) {
    prefetch_tensormap(&tmap_s);
    prefetch_tensormap(&tmap_s8);
#pragma unroll
    for (int s = 0; s < kScS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // Launched as a programmatic dependent launch, this kernel's setup above
  // overlaps the previous kernel; every global read and write comes after
  // this wait.  Then the top-k kernel may be scheduled.
  pdl_wait();
  if (tid == 0) pdl_launch_dependents();

  // ------------------------------------------------------------ producer warp
  if (warp == kScNC) {
    const bool feeder = lane < kScNC;
    const long long v = static_cast<long long>(blockIdx.x) * kScNC + lane;
    const long long e = feeder ? flat_split(v + 1, F, n_workers) : 0;
    long long f = feeder ? flat_split(v, F, n_workers) : 0;
    long long uf;
    int pos, use = 0;
    flat_divmod(f, N, uf, pos);
    bool abort = false;
    uint64_t t_prog = global_timer_ns();
#pragma unroll 1
    while (true) {
      const bool mine = f < e && !abort;
      if (!__any_sync(0xffffffffu, mine)) break;
      if (mine) {
        const int s = lane * kScR + use % kScR;
        if (use < kScR || mbar_test_wait(&empty[s], static_cast<uint32_t>((use / kScR - 1) & 1))) {
          const int cnt = sc_chunk(f, pos, N, e);
          uint8_t *dst = smem + s * kScStageBytes;
          if (cnt == kScPages) {  // four 32-page boxes
            mbar_arrive_expect_tx(&full[s], kScStageBytes);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_2d(dst + j * HALF, &tmap_s, &full[s], 64 * j, static_cast<int>(f));
          } else {  // 8-page boxes up to cnt (rows past the range are never scored out)
            const int n8 = (cnt + 7) >> 3;
            mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(n8) * 8 * kSummBytes);
            for (int r = 0; r < n8; ++r)
#pragma unroll
              for (int j = 0; j < 4; ++j)
                tma_load_2d(dst + j * HALF + r * 1024, &tmap_s8, &full[s], 64 * j,
                            static_cast<int>(f) + 8 * r);
          }
          f += cnt;
          pos += cnt;
          if (pos == N) pos = 0;
          ++use;
          t_prog = global_timer_ns();
        } else if (global_timer_ns() - t_prog > wait_ns) {
          set_status(KVR_ST_WAIT_TIMEOUT);
          s_abort = 1;
        }
        if (s_abort) abort = true;
      }
    }
    if (feeder && abort)  // never leave with copies in flight
      for (int j = max(0, use - kScR); j < use; ++j)
        mbar_wait(&full[lane * kScR + j % kScR], static_cast<uint32_t>((j / kScR) & 1), kWaitNs);
    return;
  }

  // ------------------------------------------------------------ workers
  const long long v = static_cast<long long>(blockIdx.x) * kScNC + warp;
  const long long e = flat_split(v + 1, F, n_workers);
  long long f = flat_split(v, F, n_workers);
  long long u;
  int pos;
  flat_divmod(f, N, u, pos);
  const int gq = lane >> 2, tq = lane & 3, mi = lane >> 3, mr = lane & 7;
  // [q- | q+] of row 8 cb + gq (token j / G, head j % G) as B fragments:
  // k-step kk < 8 meets kmin channels 16kk.., kk >= 8 meets kmax channels
  // 16(kk - 8)..; words hold bf16 pairs
  uint32_t qa[CB][16][2];
  long long q_unit = -1;
#pragma unroll 1
  for (int use = 0; f < e; ++use) {
    const int cnt = sc_chunk(f, pos, N, e);
    if (q_unit != u) {
      const int ui = static_cast<int>(u);  // < B H
      const int b = ui / H, g = ui - b * H;
#pragma unroll
      for (int cb = 0; cb < CB; ++cb) {
        const int jr = min(8 * cb + gq, NR - 1);
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
            q + ((static_cast<size_t>(b) * T + jr / G) * Hq + g * G + jr % G) * kD);
        const bool on = 8 * cb + gq < NR;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
          for (int hlf = 0; hlf < 2; ++hlf) {
            // q is written by no kernel that lets this one start before it
            // ends, so the read-only path is safe for it
            const uint32_t w = on ? __ldg(qrow + 8 * kk + 4 * hlf + tq) : 0u;
            // per bf16 half: all ones where the sign bit is set
            const uint32_t neg = ((w >> 15) & 0x00010001u) * 0xffffu;
            qa[cb][kk][hlf] = w & neg;        // q- with kmin
            qa[cb][8 + kk][hlf] = w & ~neg;   // q+ with kmax
          }
        }
      }
      q_unit = u;
    }
    const int s = warp * kScR + use % kScR;
    bool have = false;
    if (__shfl_sync(0xffffffffu, s_abort, 0) == 0) {  // warp-uniform
      const bool ok = mbar_wait(&full[s], static_cast<uint32_t>((use / kScR) & 1), wait_ns);
      if (__all_sync(0xffffffffu, ok)) {
        have = true;
      } else if (lane == 0) {
        s_abort = 1;
      }
    }
    if (have) {
      // S^T[page][head] on the tensor cores: pages 16 mt + gq (+8) of the
      // stage on the 16-row side, heads 2tq, 2tq + 1 as columns; even and
      // odd k-steps in separate accumulators.  Rows past cnt hold stale
      // shared memory; their results are never stored.
      const uint32_t sb = ring + s * kScStageBytes;
      float c[CB][2][4], d[CB][2][4];
#pragma unroll
      for (int cb = 0; cb < CB; ++cb)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int x = 0; x < 4; ++x) c[cb][mt][x] = d[cb][mt][x] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          uint32_t a[4];
          ldsm_x4(swz<HALF>(sb, 16 * mt + 8 * (mi & 1) + mr, 2 * kk + (mi >> 1)), a);
#pragma unroll
          for (int cb = 0; cb < CB; ++cb) {
            if (kk & 1)
              mma_bf16_16816(d[cb][mt], a[0], a[1], a[2], a[3], qa[cb][kk][0], qa[cb][kk][1]);
            else
              mma_bf16_16816(c[cb][mt], a[0], a[1], a[2], a[3], qa[cb][kk][0], qa[cb][kk][1]);
          }
        }
      // sum over the rows in a fixed order: the lane's two columns, then the
      // four column pairs (rows NR.. are zero columns), then the blocks
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float t = 0.f;
#pragma unroll
          for (int cb = 0; cb < CB; ++cb) {
            float x = (c[cb][mt][2 * r] + d[cb][mt][2 * r]) + (c[cb][mt][2 * r + 1] + d[cb][mt][2 * r + 1]);
            x += __shfl_xor_sync(0xffffffffu, x, 1);
            x += __shfl_xor_sync(0xffffffffu, x, 2);
            t = cb == 0 ? x : t + x;
          }
          t *= (1.0f / NR);
          const int p = 16 * mt + gq + 8 * r;
          if (tq == 0 && p < cnt) {
            ws_scores[f + p] = t;
            if (scores_out) scores_out[f + p] = t;
          }
        }
    }
    __syncwarp();
    // a stage is released only once its copy has landed: after an abort the
    // producer may not refill a stage whose copy is still in flight (it
    // drains those before the CTA leaves)
    if (lane == 0 && have) mbar_arrive(&empty[s]);
    f += cnt;
    pos += cnt;
    if (pos == N) {
      pos = 0;
      ++u;
    }
  }
}

// Correction decision of the speculative step, taken before (and apart from)
// the new selection, so that the attention of the reused heads does not wait
// for it (FreeKV, section 2.1: speculative retrieval takes the selection off
// the critical path).  One CTA of G warps per (b, g): warp w computes the
// cosine of q_t and q_{t-1} for query head g G + w (4 channels per lane, fp32,
// the same arithmetic as k_topk's own test), C = mean over the group,
// corrected = step == 0 or C < tau.  A reused head gets sel_used = sel_prev
// and its physical ids; q_prev <- q_t.
template <int G>
__global__ void __launch_bounds__(32 * G)
    k_spec_decide(const uint16_t *__restrict__ q, const int32_t *__restrict__ page_table, int H,
                  int N, int k, SpecArgs spec) {
  __shared__ float s_cos[G];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.x, b = blockIdx.y;
  const int Hq = H * G;
  const size_t unit = static_cast<size_t>(b) * H + g;
  const size_t qo = (static_cast<size_t>(b) * Hq + g * G + warp) * kD + 4 * lane;
  const uint2 qa = *reinterpret_cast<const uint2 *>(q + qo);
  const uint2 qb = *reinterpret_cast<const uint2 *>(spec.q_prev + qo);
  const float x[4] = {bf_lo(qa.x), bf_hi(qa.x), bf_lo(qa.y), bf_hi(qa.y)};
  const float y[4] = {bf_lo(qb.x), bf_hi(qb.x), bf_lo(qb.y), bf_hi(qb.y)};
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
  __syncthreads();
  float cb = __int_as_float(0x7fc00000);  // NaN: no previous query at step 0
  bool corrected = true;
  if (spec.step > 0) {
    float sum = 0.f;
    for (int h = 0; h < G; ++h) sum += s_cos[h];
    cb = sum / G;
    corrected = cb < spec.tau;
  }
  if (tid == 0) {
    spec.corrected[unit] = corrected ? 1 : 0;
    if (spec.cbar) spec.cbar[unit] = cb;
  }
  // q_prev <- q_t (every warp has read its head of q_prev above)
  *reinterpret_cast<uint2 *>(spec.q_prev + qo) = qa;
  if (!corrected) {  // reuse: sel_used <- previous selection, with its physical ids
    const int32_t *ptab = page_table + static_cast<size_t>(b) * N;
    for (int i = tid; i < k; i += 32 * G) {
      const int p = spec.sel_prev[unit * k + i];
      spec.sel_used[unit * k + i] = p;
      spec.sel_used_phys[unit * k + i] = (p >= 0 && p < N) ? __ldg(ptab + p) : -1;
    }
  }
}

// Selection of one (b, g) unit from its N <= NT * KPT scores, one CTA of NT
// threads (256 to 1024).  Each thread keeps KPT keys in registers: key j of lane l in warp
// w is page (w KPT + j) 32 + l, so every warp holds consecutive
// blocks of 32 pages.  The histogram rounds issue all of a thread's shared
// atomics back to back (histograms double-buffered, a round's bins cleared
// by their owners once read; the bin search is a per-warp scan plus one
// exchange of warp totals), and the ordered compaction works on ballots of
// the 32-page blocks, so no pass walks keys through shared memory.
template <int G, int NT, int KPT>
// The 512-thread, 8-key instance at 64 registers (it needs no more): its CTA
// then fits on an SM beside two scoring CTAs (30 K registers) or an
// attention CTA (24 K), so that the speculative prologue runs while the
// scores stream and a reused unit's attention starts as soon as the scoring
// ends.  (The 256-thread ones fit as they are; 16 keys would spill.)
__global__ void __launch_bounds__(NT, NT == 512 && KPT <= 8 ? 2 : 1)
    k_topk(const uint16_t *__restrict__ q, const int32_t *__restrict__ page_table, int H, int N,
           int k, const float *__restrict__ ws_scores, int32_t *__restrict__ sel_out,
           int32_t *__restrict__ sel_phys_out, SpecArgs spec,
           const int32_t *__restrict__ seq_len, int P) {
  constexpr int NW = NT / 32, BPT = kSelBins / NT;  // warps, bins per thread
  static_assert(NT % 32 == 0 && kSelBins % NT == 0, "bins are split evenly over the threads");
  __shared__ __align__(16) uint32_t s_hist[2][kSelBins];
  __shared__ uint32_t s_w1[NW], s_w2[NW];
  __shared__ uint32_t s_bin, s_bin_above, s_bin_cnt;
  __shared__ uint32_t s_cand[32], s_ncand;  // the last few keys of [L, R], ranked by one warp
  __shared__ float s_cos[8];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.x, b = blockIdx.y;
  // The kernel after this one (the attention, or the next selection) may be
  // scheduled now: its launch and setup overlap this one, and its own
  // dependency wait still covers all of this kernel's writes.
  if (tid == 0) pdl_launch_dependents();
  const int Hq = H * G;
  const size_t unit = static_cast<size_t>(b) * H + g;
  const int base = warp * KPT * 32 + lane;  // page of key j: base + 32 j
  // pages the sequence has started (all N without lengths); only these rank
  const int Nv = seq_len ? min(N, max(0, (seq_len[b] + P - 1) / P)) : N;

  // ---- speculative mode: group similarity and the correction decision,
  // taken before the wait so that it overlaps the scores kernel.  It reads
  // q_t, q_prev, sel_prev and the page table (or working-set map) and writes
  // corrected, cbar, q_prev and the reused heads' sel_used: k_page_scores,
  // the kernel this one depends on, touches none of them, and it passed its
  // own wait (so every kernel before it has finished) before letting this
  // one start.
  const int32_t *ptab = page_table ? page_table + static_cast<size_t>(b) * N : nullptr;
  bool corrected = true;
  if (spec.enabled && !spec.decided) {
    if (spec.step > 0 && warp < G) {
      const size_t qo = (static_cast<size_t>(b) * Hq + g * G + warp) * kD + 4 * lane;
      const uint2 qa = *reinterpret_cast<const uint2 *>(q + qo);
      const uint2 qb = *reinterpret_cast<const uint2 *>(spec.q_prev + qo);
      const float x[4] = {bf_lo(qa.x), bf_hi(qa.x), bf_lo(qa.y), bf_hi(qa.y)};
      const float y[4] = {bf_lo(qb.x), bf_hi(qb.x), bf_lo(qb.y), bf_hi(qb.y)};
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
    // every thread takes the same decision from the same values
    float cb = __int_as_float(0x7fc00000);  // NaN: no previous query at step 0
    if (spec.step > 0) {
      float sum = 0.f;
      for (int h = 0; h < G; ++h) sum += s_cos[h];
      cb = sum / G;
      corrected = cb < spec.tau;
    }
    if (tid == 0) {
      spec.corrected[unit] = corrected ? 1 : 0;
      if (spec.cbar) spec.cbar[unit] = cb;
    }
    // q_prev <- q_t for this group's heads (only this CTA reads them; every
    // read above is done)
    for (int i = tid; i < G * kD / 8; i += NT) {
      const size_t off = (static_cast<size_t>(b) * Hq + g * G) * kD + 8 * i;
      *reinterpret_cast<uint4 *>(spec.q_prev + off) = *reinterpret_cast<const uint4 *>(q + off);
    }
    if (!corrected) {  // reuse: sel_used <- previous selection (replaced only after the top-k)
      for (int i = tid; i < k; i += NT) {
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
    // a reused unit's page ids are final now: announce them (after every
    // thread's writes) so that its attention need not wait for this kernel
    if (spec.ready != nullptr && !corrected) {  // uniform over the CTA
      __syncthreads();
      if (tid == 0) st_release_gpu_u64(spec.ready + unit, spec.ready_tag);
    }
  }
  for (int i = tid; i < 2 * kSelBins; i += NT) (&s_hist[0][0])[i] = 0u;
  if (tid == 0) s_ncand = 0u;
  pdl_wait();  // the scores of k_page_scores are complete and visible
  if (spec.enabled && spec.decided) corrected = spec.corrected[unit] != 0;  // k_spec_decide's decision

  // the keys, all loads in flight at once, and their range
  const float *row = ws_scores + unit * N;
  float sv[KPT];
#pragma unroll
  // at L2, never through the read-only path: k_page_scores writes them while
  // this kernel is already resident (programmatic dependent launch), so a
  // read-only cache could still hold an earlier call's lines
  for (int j = 0; j < KPT; ++j) sv[j] = base + 32 * j < Nv ? __ldcg(row + base + 32 * j) : 0.f;
  uint32_t key[KPT];
  uint32_t kmn = 0xffffffffu, kmx = 0u;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    key[j] = score_key(sv[j]);
    if (base + 32 * j < Nv) {
      kmn = min(kmn, key[j]);
      kmx = max(kmx, key[j]);
    }
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    kmn = min(kmn, __shfl_xor_sync(0xffffffffu, kmn, m));
    kmx = max(kmx, __shfl_xor_sync(0xffffffffu, kmx, m));
  }
  if (lane == 0) {
    s_w1[warp] = kmn;
    s_w2[warp] = kmx;
  }
  // page-table entries of this thread's pages, for the physical ids of the
  // selected ones, in flight during the histogram rounds (issued after the
  // scores, which are on the critical path)
  const bool want_phys = spec.enabled ? (spec.sel_used_phys && !spec.page2slot && (spec.decided || corrected))
                                      : sel_phys_out != nullptr;
  int phys[KPT];
#pragma unroll
  for (int j = 0; j < KPT; ++j) phys[j] = want_phys && base + 32 * j < Nv ? __ldg(ptab + base + 32 * j) : -1;
  __syncthreads();
  uint32_t L = 0xffffffffu, R = 0u;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    L = min(L, s_w1[w]);
    R = max(R, s_w2[w]);
  }
  // invariant: `need` of the `cnt` keys in [L, R] are still to be taken;
  // every key above R is taken
  const int n_take = min(k, Nv);  // keys selected in all (slots 0 .. n_take-1)
  uint32_t need = static_cast<uint32_t>(n_take), cnt = static_cast<uint32_t>(Nv);
  int buf = 0;
#pragma unroll 1
  while (cnt != need && L != R) {
    if (cnt <= 32u) {
      // few keys left in [L, R] (usually after one round): one warp ranks
      // them instead of another histogram pass.  The need-th largest value v
      // of the interval has gt keys above it and eq equal to it, with
      // gt < need <= gt + eq; then L = R = v, and need - gt of the eq keys
      // equal to v are taken (the first by page id, in the compaction).
#pragma unroll
      for (int j = 0; j < KPT; ++j)
        if (base + 32 * j < Nv && key[j] >= L && key[j] <= R) s_cand[atomicAdd(&s_ncand, 1u)] = key[j];
      __syncthreads();
      if (warp == 0) {
        const uint32_t c = s_ncand;  // == cnt
        const uint32_t mine = lane < static_cast<int>(c) ? s_cand[lane] : 0u;
        uint32_t gt = 0u, eq = 0u;
        for (uint32_t o = 0; o < c; ++o) {
          const uint32_t x = __shfl_sync(0xffffffffu, mine, static_cast<int>(o));
          gt += x > mine ? 1u : 0u;
          eq += x == mine ? 1u : 0u;
        }
        if (lane < static_cast<int>(c) && gt < need && need <= gt + eq) {  // lanes of v write the same
          s_bin = mine;
          s_bin_above = gt;
          s_bin_cnt = eq;
        }
      }
      __syncthreads();
      L = R = s_bin;
      need -= s_bin_above;
      cnt = s_bin_cnt;
      break;
    }
    const uint32_t span = R - L;
    const int shift = span < kSelBins ? 0 : (32 - __clz(span)) - 11;
    uint32_t *hist = s_hist[buf];
#pragma unroll
    for (int j = 0; j < KPT; ++j)
      if (base + 32 * j < Nv && key[j] >= L && key[j] <= R)
        atomicAdd(&hist[(key[j] - L) >> shift], 1u);
    __syncthreads();
    // thread tid owns bins [BPT tid, BPT tid + BPT); clear them for the round
    // after next once read
    // (vector accesses: a quarter warp covers 128 contiguous bytes)
    uint32_t c[BPT], mine = 0u;
    if constexpr (BPT % 4 == 0) {
      uint4 *hv = reinterpret_cast<uint4 *>(hist + BPT * tid);
#pragma unroll
      for (int v = 0; v < BPT / 4; ++v) {
        const uint4 x = hv[v];
        hv[v] = make_uint4(0u, 0u, 0u, 0u);
        c[4 * v] = x.x;
        c[4 * v + 1] = x.y;
        c[4 * v + 2] = x.z;
        c[4 * v + 3] = x.w;
      }
    } else {
      static_assert(BPT == 2, "bins per thread");
      uint2 *hv = reinterpret_cast<uint2 *>(hist + BPT * tid);
      const uint2 x = hv[0];
      hv[0] = make_uint2(0u, 0u);
      c[0] = x.x;
      c[1] = x.y;
    }
#pragma unroll
    for (int e = 0; e < BPT; ++e) mine += c[e];
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_w1[warp] = incl;
    __syncthreads();
    uint32_t total = 0u, before = 0u;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const uint32_t x = s_w1[w];
      total += x;
      before += w < warp ? x : 0u;
    }
    uint32_t above_here = total - (before + incl);  // keys of the interval in higher bins
#pragma unroll
    for (int e = BPT - 1; e >= 0; --e) {
      if (above_here < need && need <= above_here + c[e]) {
        s_bin = static_cast<uint32_t>(BPT * tid + e);
        s_bin_above = above_here;
        s_bin_cnt = c[e];
      }
      above_here += c[e];
    }
    __syncthreads();
    const uint32_t nl = L + (s_bin << shift);
    const unsigned long long nr = static_cast<unsigned long long>(nl) + ((1ull << shift) - 1ull);
    need -= s_bin_above;
    cnt = s_bin_cnt;
    R = static_cast<uint32_t>(min(static_cast<unsigned long long>(R), nr));
    L = nl;
    buf ^= 1;
  }

  // ---- ordered compaction (ascending page ids): every key above R, then the
  // first `need` keys of [L, R] by page id (all of them when cnt == need).
  // Per 32-page block: ballots of the two kinds; per warp: running counts;
  // across warps: one exchange of the warp totals.
  const uint32_t lt = (1u << lane) - 1u;  // lanes below this one
  // the warp's counts of the two kinds: this lane's counts, summed over lanes
  uint32_t w_gt = 0u, w_eq = 0u;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const bool valid = base + 32 * j < Nv;
    w_gt += (valid && key[j] > R) ? 1u : 0u;
    w_eq += (valid && key[j] >= L && key[j] <= R) ? 1u : 0u;
  }
  w_gt |= w_eq << 16;  // both counts (<= 32 KPT each) in one word
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) w_gt += __shfl_xor_sync(0xffffffffu, w_gt, m);
  w_eq = w_gt >> 16;
  w_gt &= 0xffffu;
  __syncthreads();  // s_w* free; every read of the previous selection is done
  if (lane == 0) {
    s_w1[warp] = w_gt;
    s_w2[warp] = w_eq;
  }
  __syncthreads();
  uint32_t gt_seen = 0u, eq_seen = 0u;  // keys of the two kinds in lower pages
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    gt_seen += w < warp ? s_w1[w] : 0u;
    eq_seen += w < warp ? s_w2[w] : 0u;
  }
  int pos[KPT];
  int nsel = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {  // the ballots again, now in page order
    const bool valid = base + 32 * j < Nv;
    const bool is_gt = valid && key[j] > R, is_eq = valid && key[j] >= L && key[j] <= R;
    const uint32_t m_gt = __ballot_sync(0xffffffffu, is_gt);
    const uint32_t m_eq = __ballot_sync(0xffffffffu, is_eq);
    const uint32_t gb = gt_seen + __popc(m_gt & lt), eb = eq_seen + __popc(m_eq & lt);
    const bool take = is_gt || (is_eq && eb < need);
    const uint32_t out = gb + min(eb, need);  // selected keys in lower pages
    pos[j] = take && out < static_cast<uint32_t>(k) ? static_cast<int>(out) : -1;
    nsel += pos[j] >= 0;
    gt_seen += __popc(m_gt);
    eq_seen += __popc(m_eq);
  }
  // fewer started pages than k (lengths only): slots n_take .. k-1, which no
  // selected key takes, are -1
  if (!spec.enabled)
    for (int i = n_take + tid; i < k; i += NT) {
      sel_out[unit * k + i] = -1;
      if (sel_phys_out) sel_phys_out[unit * k + i] = -1;
    }
  if (nsel == 0) return;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    if (pos[j] < 0) continue;
    const int i = base + 32 * j;
    const size_t o = unit * k + pos[j];
    if (spec.enabled) {
      spec.sel_prev[o] = i;
      if (corrected) {
        spec.sel_used[o] = i;
        if (want_phys) spec.sel_used_phys[o] = phys[j];
      }
    } else {
      sel_out[o] = i;
      if (want_phys) sel_phys_out[o] = phys[j];
    }
  }
}

}  // namespace kvr
