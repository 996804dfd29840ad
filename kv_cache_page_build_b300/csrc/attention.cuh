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
// Work decomposition.  Unit u is handled by one cluster of Q CTAs (Q in
// {1, 2, 4, 8}, chosen on the host so that the Q x units CTAs are resident
// together when they fit).  The unit's k CPP chunks of C = min(P, 32) tokens
// are cut into Q NC equal contiguous ranges, one per consumer warp (a
// "worker") of the cluster.  A worker keeps its split's running (m, l, O) in
// registers; at the end it stages O in one of its own (now idle) ring stages
// and pushes it, 16 bytes per store through distributed shared memory, to
// the CTAs that merge it: CTA r merges channels [r D/Q, (r+1) D/Q) of the G
// heads, and every CTA gets every worker's (m, l).  After one cluster
// barrier each CTA merges its slice from its own shared memory with a
// log-sum-exp rescale and writes it to `out`; no CTA reads another's shared
// memory after the barrier, so each leaves as soon as it is done.  Before the
// first push, a handshake (every thread arrives right after the setup and
// waits before pushing) makes sure every CTA of the cluster has started, as
// distributed shared memory requires.  Nothing of
// the split goes through global memory and no second kernel is needed.
//
// Inside a CTA (CPS per SM) the warps share the shared-memory ring:
//   producer  warp NC; lane w feeds consumer warp w, which owns R stages of
//        the ring: as soon as the warp releases a stage, the lane issues the
//        warp's next chunk into it (four tiled TMA copies: the 64-channel
//        halves of the chunk's K and V rows for head g, 128-byte swizzled).
//        The ranges' page ids are read into shared memory first, so issuing
//        never waits on a load.
//   consumer  warps 0..NC-1 on the tensor cores (mma.sync m16n8k16, bf16 in,
//        fp32 accumulators), one chunk at a time (attn_chunk): S^T = K q^T
//        with the chunk's tokens on the MMA's 16-row side, online softmax in
//        base 2, then O^T += V^T P^T with P^T moved into the operand layout
//        by movmatrix and split into a bf16 high part and residual.
// The G x D output of a group is a 4- to 32-row contraction per page, far
// from the tensor cores' peak; they are used because they cut the issue
// slots per chunk several-fold against CUDA-core FMAs, which keeps the
// consumers ahead of the memory stream.
// Every wait on a copy is bounded; after a timeout the CTA stops issuing
// copies, drains the ones in flight and still takes part in the cluster
// barrier, which every thread of the cluster reaches after bounded work.
#pragma once

#include "common.cuh"

namespace kvr {

constexpr int kAttnNC = 4;                         // consumer warps per CTA
constexpr int kAttnThreads = 32 * (kAttnNC + 1);   // + one producer warp
constexpr int kAttnIds = 128;                      // page ids of a worker range kept in shared memory
constexpr int kAttnCPS = 1;                        // CTAs per SM
constexpr int kAttnMaxQ = 8;                       // CTAs per cluster (the portable limit)
constexpr int kAttnWarpRing = 48 * 1024;           // ring bytes of one consumer warp
constexpr int kSmemPerSM = 228 * 1024;             // shared memory of one SM

// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32: relative error
// about 2^-22; 2^-inf = +0), for the softmax weights and the merge's rescale.
// Against exp2f it takes fewer instructions on the consumers' path, which
// the memory stream waits on.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// NR: query rows per unit, the G heads of the group times the T query tokens
// of the step (1, 2, 4, 8 or 16); they are the MMA's column side, in CB
// blocks of 8 columns.
template <int NR, int P>
struct AttnCfg {
  static constexpr int CB = NR > 8 ? 2 : 1;        // 8-column blocks of the query rows
  static constexpr int C = P < 32 ? P : 32;        // tokens per chunk (one stage)
  static constexpr int CPP = P / C;                // chunks per page
  static constexpr int NB = C / 8;                 // 8-token column blocks of the QK MMA
  static constexpr int KP = C / 16;                // 16-token k-steps of the PV MMA
  static constexpr int kHalf = C * 128;            // 64 channels of C rows (swizzled)
  static constexpr int kStageBytes = 4 * kHalf;    // K lo, K hi, V lo, V hi
  // ring bytes of one consumer warp: 48 KiB, 32 KiB with two column blocks
  // (whose partials need twice the receive space)
  static constexpr int kWarpRing = CB == 1 ? kAttnWarpRing : 32 * 1024;
  static constexpr int R = kWarpRing / kStageBytes;  // stages per consumer warp
  static constexpr int S = kAttnNC * R;            // ring depth
  static constexpr int kSmem = S * kStageBytes + 1024;   // + 1 KiB to align the ring
  static constexpr int kStatic = kAttnNC * NR * kD * 4 + kAttnMaxQ * kAttnNC * NR * 8 +
                                 2 * kAttnNC * kAttnIds * 4 + S * 28 + 64;
  static_assert(kAttnCPS * (kSmem + kStatic + 1024) <= kSmemPerSM, "CTAs per SM must fit");
  static_assert(CPP * C == P && NB * 8 == C && KP * 16 == C && R >= 2, "chunk tiling");
  static_assert(NR * kD * 4 + NR * 8 <= R * kStageBytes, "a worker's partial fits its stages");
};

__device__ __forceinline__ bool attn_unit_active(const uint8_t *filter, int filter_mode,
                                                 long long u) {
  if (filter_mode == 0) return true;
  return (filter[u] != 0) == (filter_mode == 2);
}

// One chunk of C tokens for a consumer warp.
//   QK   S^T[t][j] = K_t . q_j with the tokens on the MMA's 16-row side and
//        the query rows as its columns (8 per block; rows NR.. are zero):
//        C/16 row blocks x 8 channel k-steps per column block; K fragments
//        by ldmatrix, q as B fragments held in registers.  Lane (gq, tq)
//        gets tokens 16 mt + gq (+8) of columns 8 cb + 2tq, 8 cb + 2tq + 1.
//   softmax  online, base 2 (logits prescaled by scale * log2 e); the lane's
//        running (m, l) are those of its columns.
//   PV   O^T[c][j] += V^T[c][t] P^T[t][j]: V fragments by transposing
//        ldmatrix; P^T as B fragments by transposing the accumulator tiles
//        in registers (movmatrix).  P is split into a bf16 high part and a
//        bf16 residual, so the weights keep about 16 bits: for NR <= 4 the
//        residual rides in columns j + 4 of the same MMA (the output of row
//        j is then column j plus column j + 4); otherwise it takes a second
//        MMA.
// nv: tokens of the chunk that exist (C except in the partial last page of
// a sequence): their V rows beyond nv are zeroed, so stale rows can
// contribute neither weight nor NaN.  lim[cb][c]: the leading tokens of the
// chunk that the lane's column 8 cb + 2tq + c may see (at most nv; fewer for
// an earlier query token of the step, which attends causally); the scores of
// the others become -inf.  A column that has seen no token yet keeps
// m = -inf and l = 0.
template <int NR, int P, bool CAUSAL>
__device__ __forceinline__ void attn_chunk(uint32_t kb, const uint32_t (&qb)[AttnCfg<NR, P>::CB][8][2],
                                           float scale_log2, float (&m_run)[AttnCfg<NR, P>::CB][2],
                                           float (&l_run)[AttnCfg<NR, P>::CB][2],
                                           float (&o)[AttnCfg<NR, P>::CB][8][4], int lane, int nv,
                                           const int (&lim)[AttnCfg<NR, P>::CB][2]) {
  using Cfg = AttnCfg<NR, P>;
  constexpr int HALF = Cfg::kHalf, MT = Cfg::C / 16, CB = Cfg::CB;
  constexpr bool kPair = NR <= 4;
  const int gq = lane >> 2, tq = lane & 3, mi = lane >> 3, mr = lane & 7;
  const uint32_t vb = kb + 2 * HALF;
  if (nv < Cfg::C) {  // zero V rows nv .. C-1 of both channel halves (16 bytes a lane-store)
    for (int x = lane; x < (Cfg::C - nv) * 16; x += 32) {
      const int row = nv + (x >> 4), half = (x >> 3) & 1, chunk = x & 7;
      asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vb + half * HALF + row * 128 + chunk * 16),
                   "r"(0u)
                   : "memory");
    }
    __syncwarp();
  }
  // ---- S^T, even and odd channel k-steps in separate accumulators
  float st[CB][MT][4], su[CB][MT][4];
#pragma unroll
  for (int cb = 0; cb < CB; ++cb)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) st[cb][mt][e] = su[cb][mt][e] = 0.f;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      uint32_t a[4];
      ldsm_x4(swz<HALF>(kb, 16 * mt + 8 * (mi & 1) + mr, 2 * kk + (mi >> 1)), a);
#pragma unroll
      for (int cb = 0; cb < CB; ++cb) {
        if (kk & 1)
          mma_bf16_16816(su[cb][mt], a[0], a[1], a[2], a[3], qb[cb][kk][0], qb[cb][kk][1]);
        else
          mma_bf16_16816(st[cb][mt], a[0], a[1], a[2], a[3], qb[cb][kk][0], qb[cb][kk][1]);
      }
    }
  uint32_t pb[CB][MT][2], pl[CB][MT][2];
#pragma unroll
  for (int cb = 0; cb < CB; ++cb) {
    // ---- online softmax for columns 8 cb + 2tq (e = 0, 2) and + 1 (e = 1, 3)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        st[cb][mt][e] = (st[cb][mt][e] + su[cb][mt][e]) * scale_log2;
        if (16 * mt + gq + 8 * (e >> 1) >= (CAUSAL ? lim[cb][e & 1] : nv))
          st[cb][mt][e] = -INFINITY;  // not visible
      }
      mx0 = fmaxf(mx0, fmaxf(st[cb][mt][0], st[cb][mt][2]));
      mx1 = fmaxf(mx1, fmaxf(st[cb][mt][1], st[cb][mt][3]));
    }
#pragma unroll
    for (int m = 4; m <= 16; m <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, m));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, m));
    }
    const float mn0 = fmaxf(m_run[cb][0], mx0), mn1 = fmaxf(m_run[cb][1], mx1);
    // exponent base: 0 while a column has seen no token (everything is -inf;
    // without the causal limits every column sees the chunk's first token)
    const float mb0 = CAUSAL && mn0 == -INFINITY ? 0.f : mn0;
    const float mb1 = CAUSAL && mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = ex2_approx(m_run[cb][0] - mb0), al1 = ex2_approx(m_run[cb][1] - mb1);
    const bool on0 = 8 * cb + 2 * tq < NR, on1 = 8 * cb + 2 * tq + 1 < NR;
    float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      st[cb][mt][0] = on0 ? ex2_approx(st[cb][mt][0] - mb0) : 0.f;
      st[cb][mt][2] = on0 ? ex2_approx(st[cb][mt][2] - mb0) : 0.f;
      st[cb][mt][1] = on1 ? ex2_approx(st[cb][mt][1] - mb1) : 0.f;
      st[cb][mt][3] = on1 ? ex2_approx(st[cb][mt][3] - mb1) : 0.f;
      ls0 += st[cb][mt][0] + st[cb][mt][2];
      ls1 += st[cb][mt][1] + st[cb][mt][3];
    }
    l_run[cb][0] = fmaf(l_run[cb][0], al0, ls0);
    l_run[cb][1] = fmaf(l_run[cb][1], al1, ls1);
    m_run[cb][0] = mn0;
    m_run[cb][1] = mn1;
    // rescale O; with the residual in columns j + 4, lanes tq >= 2 hold the
    // residual columns of rows 2tq - 4, 2tq - 3 (the lane tq - 2's rows)
    float a0 = al0, a1 = al1;
    if (kPair) {
      const float x0 = __shfl_xor_sync(0xffffffffu, al0, 2);
      const float x1 = __shfl_xor_sync(0xffffffffu, al1, 2);
      if (tq >= 2) {
        a0 = x0;
        a1 = x1;
      }
    }
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      o[cb][mb][0] *= a0;
      o[cb][mb][1] *= a1;
      o[cb][mb][2] *= a0;
      o[cb][mb][3] *= a1;
    }
    // ---- P^T as B fragments: 8x8 tiles (tokens 16 mt + 8 r .., columns) transposed
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float x0 = st[cb][mt][2 * r], x1 = st[cb][mt][2 * r + 1];
        const uint32_t hi = pack_bf16x2(x0, x1);
        const uint32_t lo = pack_bf16x2(x0 - __uint_as_float(hi << 16),
                                        x1 - __uint_as_float(hi & 0xffff0000u));
        if (kPair) {
          const uint32_t lo_s = __shfl_xor_sync(0xffffffffu, lo, 2);
          pb[cb][mt][r] = movmatrix_trans(tq < 2 ? hi : lo_s);
          pl[cb][mt][r] = 0u;
        } else {
          pb[cb][mt][r] = movmatrix_trans(hi);
          pl[cb][mt][r] = movmatrix_trans(lo);
        }
      }
  }
  // ---- PV: O^T[16 mb ..][columns] += V^T[16 mb ..][16 kp ..] P^T
#pragma unroll
  for (int mb = 0; mb < 8; ++mb) {
#pragma unroll
    for (int kp = 0; kp < MT; ++kp) {
      uint32_t va[4];
      ldsm_x4_trans(swz<HALF>(vb, 16 * kp + 8 * (mi >> 1) + mr, 2 * mb + (mi & 1)), va);
#pragma unroll
      for (int cb = 0; cb < CB; ++cb) {
        mma_bf16_16816(o[cb][mb], va[0], va[1], va[2], va[3], pb[cb][kp][0], pb[cb][kp][1]);
        if (!kPair) mma_bf16_16816(o[cb][mb], va[0], va[1], va[2], va[3], pl[cb][kp][0], pl[cb][kp][1]);
      }
    }
  }
}

// filter_mode: 0 every unit; 1 only units with filter[unit] == 0; 2 only != 0.
// Grid: units x Q CTAs in clusters of Q (cluster c = unit c).
// T query tokens per sequence and G query heads per KV head (NR = T G): q and
// out are [B][T][Hq][D]; with T > 1 seq_len and sel_log (the logical ids of
// sel_phys) are given and query token tau sees the positions below
// seq_len - T + tau + 1 (CAUSAL instances; T = 1 takes the others).  out is
// fp32, or bf16 (rounded to nearest even) when out_bf16 != 0.
// ready (may be null; speculative step, every unit active): a unit whose
// word holds ready_tag when its CTA starts had its page ids written and
// announced by the top-k kernel before that kernel finished (a reused
// selection): the CTA starts at once and waits for the kernel it depends on
// only before it leaves.  The ids are read at L2 (never through the
// read-only path, as they may have been written during this kernel's
// lifetime).  CTA 0 of the cluster clears the word at the end.
// Register cap: at most 128 per thread for up to 8 query rows (they need
// 127 and do not spill), so that an attention CTA (5 warps) fits on an SM
// beside a 512-thread top-k CTA: each SM sub-partition's 16 K registers then
// hold its four top-k warps (4 x 2048) and up to two attention warps
// (2 x 4096); at 146 registers they did not, and the attention CTAs of a
// speculative step that land there could not start before the top-k ended.
// 16 rows keep their registers (they would spill).  kAttnCPS CTAs per SM.
template <int NR, int P, bool CAUSAL>
__global__ void __maxnreg__(NR <= 8 ? 128 : 255)
    k_sparse_decode(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const uint16_t *__restrict__ q,
                    const int32_t *__restrict__ sel_phys, const int32_t *__restrict__ sel_log,
                    int H, int k, int n_phys, int Q, int T, int G, float scale_log2, uint64_t wait_ns,
                    const uint8_t *__restrict__ filter, int filter_mode, void *__restrict__ out,
                    int out_bf16, const int32_t *__restrict__ seq_len,
                    const int32_t *__restrict__ page_table, int N,
                    unsigned long long *__restrict__ ready, unsigned long long ready_tag) {
  using Cfg = AttnCfg<NR, P>;
  constexpr int NC = kAttnNC, CPP = Cfg::CPP, HALF = Cfg::kHalf, R = Cfg::R, S = Cfg::S, CB = Cfg::CB;
  constexpr int kIdRounds = kAttnIds / 32;
  extern __shared__ uint8_t smem_raw[];
  // the swizzle pattern repeats every 1024 bytes: align the ring to it
  uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  const uint32_t ring = smem_addr(smem);
  __shared__ __align__(8) uint64_t full[S], empty[S];
  __shared__ int s_ok[S];
  __shared__ int s_nv[S];    // tokens of the stage's chunk that exist
  __shared__ int s_pos0[S];  // position of the chunk's first token in its sequence (T > 1)
  __shared__ int s_ids[NC][kAttnIds];   // page ids of the first kAttnIds chunks of each worker
  __shared__ int s_lids[NC][kAttnIds];  // their logical ids (T > 1)
  // partials of the cluster's workers for this CTA's channel slice:
  // [worker][query row][channel of the slice], and (m, l) per worker and row
  __shared__ __align__(16) float s_recv[NC * NR * kD];
  __shared__ __align__(8) float2 s_mlr[kAttnMaxQ * NC * NR];
  __shared__ volatile int s_abort;
  __shared__ int s_early;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = cluster_ctarank();
  // 32-bit index arithmetic throughout (64-bit divisions are emulated and
  // sat on the path to the first copy): u < B H, k CPP <= 2 kMaxPages and
  // the worker count is at most 32, so every product below fits
  const int u = static_cast<int>(blockIdx.x) / Q;
  const int b = u / H, g = u - b * H;
  const int nw = Q * NC;                                  // workers of the unit
  const int per = kD / Q;                                 // channels merged by each CTA
  const int kc = k * CPP;                                 // chunks of the unit
  const int32_t *sel_u = sel_phys + static_cast<size_t>(u) * k;  // the unit's page ids
  constexpr bool causal = CAUSAL;  // T > 1: seq_len and sel_log are given
  // heads per KV head: NR itself for one query token (a compile-time constant)
  const int Gc = CAUSAL ? G : NR;
  const int32_t *sel_lu = causal ? sel_log + static_cast<size_t>(u) * k : nullptr;
  // range of this CTA's worker w: chunks [a, a + n) of the unit
  auto worker_range = [&](int w, int &a, int &n) {
    const uint32_t v = static_cast<uint32_t>(rank * NC + w);
    a = static_cast<int>(v * static_cast<uint32_t>(kc) / static_cast<uint32_t>(nw));
    n = static_cast<int>((v + 1) * static_cast<uint32_t>(kc) / static_cast<uint32_t>(nw)) - a;
  };

  if (tid == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
#pragma unroll
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    s_abort = 0;
    s_early = ready != nullptr && ld_acquire_gpu_u64(ready + u) == ready_tag;
    fence_barrier_init();
  }
  __syncthreads();
  // Launched as a programmatic dependent launch, the setup above overlaps
  // the previous kernel; every global read and write comes after this wait,
  // except in an early unit (its inputs were announced; it waits at the end).
  // The next kernel may be scheduled at once: its own wait covers this one.
  const bool early = s_early != 0;
  if (tid == 0) pdl_launch_dependents();
  if (!early) pdl_wait();
  // the whole cluster holds one unit, so this exit is uniform over it (no
  // thread of the cluster touches another CTA's shared memory)
  if (!attn_unit_active(filter, filter_mode, u)) {
    if (early) pdl_wait();
    return;
  }
  // Start handshake of the cluster: no thread may write another CTA's shared
  // memory before that CTA has started; every thread arrives here and waits
  // (cluster_wait) before the first push of the merge.
  cluster_arrive_relaxed();

  if (warp == NC) {
    // ---------------------------------------------------------- producer warp
    // page ids of the workers' ranges, once (all loads in flight together),
    // so that issuing never waits on a load
    {
      int idv[NC][kIdRounds];
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        int a, n;
        worker_range(w, a, n);
#pragma unroll
        for (int r = 0; r < kIdRounds; ++r) {
          const int j = lane + 32 * r;
          idv[w][r] = j < n ? __ldcg(sel_u + (a + j) / CPP) : -1;
        }
      }
#pragma unroll
      for (int w = 0; w < NC; ++w)
#pragma unroll
        for (int r = 0; r < kIdRounds; ++r) s_ids[w][lane + 32 * r] = idv[w][r];
      if (causal) {
#pragma unroll
        for (int w = 0; w < NC; ++w) {
          int a, n;
          worker_range(w, a, n);
#pragma unroll
          for (int r = 0; r < kIdRounds; ++r) {
            const int j = lane + 32 * r;
            idv[w][r] = j < n ? __ldcg(sel_lu + (a + j) / CPP) : -1;
          }
        }
#pragma unroll
        for (int w = 0; w < NC; ++w)
#pragma unroll
          for (int r = 0; r < kIdRounds; ++r) s_lids[w][lane + 32 * r] = idv[w][r];
      }
    }
    __syncwarp();
    // with lengths, only the sequence's last page can be partial: its
    // physical id and written tokens (-1 ids are padding, skipped silently)
    int last_phys = -2, last_nt = P, L = 0;
    if (seq_len) {
      L = seq_len[b];
      if (L > 0) {
        const int pl = (L - 1) / P;
        last_phys = pl < N ? __ldg(page_table + static_cast<size_t>(b) * N + pl) : -2;
        last_nt = L - pl * P;
      }
    }
    // lane w (< NC) feeds consumer warp w: the worker's chunks go to its R
    // stages in turn
    const bool feeder = lane < NC;
    int a = 0, n = 0;
    if (feeder) worker_range(lane, a, n);
    int i = 0;
    bool abort = false;
    uint64_t t_prog = global_timer_ns();
#pragma unroll 1
    while (true) {
      const bool mine = i < n && !abort;
      if (!__any_sync(0xffffffffu, mine)) break;
      if (mine) {
        const int s = lane * R + i % R;
        if (i < R || mbar_test_wait(&empty[s], static_cast<uint32_t>((i / R - 1) & 1))) {
          const int pos = a + i;
          const int id = i < kAttnIds ? s_ids[lane][i] : __ldcg(sel_u + pos / CPP);
          int nv, pos0 = 0;
          if (causal) {  // tokens below the sequence's length, from the logical position
            const int lid = i < kAttnIds ? s_lids[lane][i] : __ldcg(sel_lu + pos / CPP);
            pos0 = lid * P + (pos % CPP) * Cfg::C;
            nv = lid >= 0 ? min(Cfg::C, max(0, L - pos0)) : 0;
          } else {
            nv = id == last_phys ? min(Cfg::C, max(0, last_nt - (pos % CPP) * Cfg::C)) : Cfg::C;
          }
          const bool ok = id >= 0 && id < n_phys && nv > 0;
          s_ok[s] = ok ? 1 : 0;
          s_nv[s] = nv;
          if (causal) s_pos0[s] = pos0;
          if (ok) {
            uint8_t *dst = smem + s * Cfg::kStageBytes;
            const int row = id * P + (pos % CPP) * Cfg::C;
            mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
            tma_load_3d(dst, &tmap_k, &full[s], 0, g, row);
            tma_load_3d(dst + HALF, &tmap_k, &full[s], 64, g, row);
            tma_load_3d(dst + 2 * HALF, &tmap_v, &full[s], 0, g, row);
            tma_load_3d(dst + 3 * HALF, &tmap_v, &full[s], 64, g, row);
          } else {
            if (nv > 0 && !(seq_len && id == -1)) set_status(KVR_ST_BAD_INDEX);
            mbar_arrive(&full[s]);
          }
          ++i;
          t_prog = global_timer_ns();
        } else if (global_timer_ns() - t_prog > wait_ns) {
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
        mbar_wait(&full[lane * R + j % R], static_cast<uint32_t>((j / R) & 1), kWaitNs);
    __syncwarp();
    cluster_wait();  // the start handshake's second half (see above)
  } else {
    // ---------------------------------------------------------- consumer warps
    const int cw = warp;
    const int gq = lane >> 2, tq = lane & 3;  // MMA fragment row group and column pair
    const int Hq = H * Gc;
    int a, n;
    worker_range(cw, a, n);
    const int L = causal ? seq_len[b] : 0;

    // query row j = 8 cb + gq (token j / G, head j % G of the group) as B
    // fragments (k-step kk: channels 16kk + 2tq, +8); rows NR.. are zero
    uint32_t qb[CB][8][2];
    float m_run[CB][2], l_run[CB][2];  // columns 8 cb + 2tq, + 1
    float o[CB][8][4];                 // O^T[16 mb + gq (+8)][8 cb + 2 tq (+1)]
#pragma unroll
    for (int cb = 0; cb < CB; ++cb) {
      m_run[cb][0] = m_run[cb][1] = -INFINITY;
      l_run[cb][0] = l_run[cb][1] = 0.f;
#pragma unroll
      for (int mb = 0; mb < 8; ++mb) o[cb][mb][0] = o[cb][mb][1] = o[cb][mb][2] = o[cb][mb][3] = 0.f;
      const int jr = min(8 * cb + gq, NR - 1);
      const int tau = CAUSAL ? jr / Gc : 0;  // one query token: row jr is head jr
      const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
          q + ((static_cast<size_t>(b) * T + tau) * Hq + g * Gc + jr - tau * Gc) * kD);
      const bool on = 8 * cb + gq < NR;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qb[cb][kk][0] = on ? __ldg(qrow + 8 * kk + tq) : 0u;
        qb[cb][kk][1] = on ? __ldg(qrow + 8 * kk + 4 + tq) : 0u;
      }
    }
#pragma unroll 1
    for (int i = 0; i < n; ++i) {
      const int s = cw * R + i % R;  // this warp's stages in turn
      // a chunk that has landed is taken at once; only a wait looks at the
      // abort flag first (after an abort nothing more lands), then waits
      // with the bound in force (warp-uniform throughout)
      bool landed = __all_sync(0xffffffffu, mbar_try_wait(&full[s], static_cast<uint32_t>((i / R) & 1)));
      if (!landed && __shfl_sync(0xffffffffu, s_abort, 0) == 0) {
        const bool ok = mbar_wait(&full[s], static_cast<uint32_t>((i / R) & 1), wait_ns);
        if (__all_sync(0xffffffffu, ok))
          landed = true;
        else if (lane == 0)
          s_abort = 1;
      }
      const bool have = landed && s_ok[s] != 0;
      if (have) {
        const int nv = s_nv[s];
        int lim[CB][2];
#pragma unroll
        for (int cb = 0; cb < CB; ++cb)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            lim[cb][c] = nv;
            if (causal) {  // query token tau sees positions below L - T + tau + 1
              const int tau = min(8 * cb + 2 * tq + c, NR - 1) / Gc;
              lim[cb][c] = min(nv, max(0, L - T + tau + 1 - s_pos0[s]));
            }
          }
        attn_chunk<NR, P, CAUSAL>(ring + s * Cfg::kStageBytes, qb, scale_log2, m_run, l_run, o, lane, nv, lim);
      }
      __syncwarp();
      // a stage is released only once its copy has landed: after an abort
      // the producer may not refill a stage whose copy is still in flight
      // (it drains those before the CTA leaves)
      if (lane == 0 && landed) mbar_arrive(&empty[s]);
    }
    // ---- this worker's partial, pushed to the CTAs that merge it
    float lr[CB][2];
#pragma unroll
    for (int cb = 0; cb < CB; ++cb)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float x = l_run[cb][c];
#pragma unroll
        for (int m = 4; m <= 16; m <<= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
        lr[cb][c] = x;
      }
    if (NR <= 4) {  // add the residual columns j + 4 into columns j
#pragma unroll
      for (int mb = 0; mb < 8; ++mb)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[0][mb][e] += __shfl_xor_sync(0xffffffffu, o[0][mb][e], 2);
    }
    // stage O [row][channel] and (m, l) [row] in this warp's first stages,
    // free now that its last chunk is consumed
    float *stg = reinterpret_cast<float *>(smem + cw * R * Cfg::kStageBytes);
    float2 *stg_ml = reinterpret_cast<float2 *>(stg + NR * kD);
#pragma unroll
    for (int cb = 0; cb < CB; ++cb)
#pragma unroll
      for (int mb = 0; mb < 8; ++mb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int jr = 8 * cb + 2 * tq + (e & 1);
          if (jr < NR) stg[jr * kD + 16 * mb + gq + 8 * (e >> 1)] = o[cb][mb][e];
        }
    if (gq == 0) {
#pragma unroll
      for (int cb = 0; cb < CB; ++cb) {
        if (8 * cb + 2 * tq < NR) stg_ml[8 * cb + 2 * tq] = make_float2(m_run[cb][0], lr[cb][0]);
        if (8 * cb + 2 * tq + 1 < NR) stg_ml[8 * cb + 2 * tq + 1] = make_float2(m_run[cb][1], lr[cb][1]);
      }
    }
    __syncwarp();
    cluster_wait();  // every CTA of the cluster has started: pushes may begin
    const int j = rank * NC + cw;  // this worker's index in the cluster
    const uint32_t rc0 = smem_addr(s_recv), ml0 = smem_addr(s_mlr);
#pragma unroll
    for (int x = lane; x < NR * kD / 4; x += 32) {  // 4 channels of one row per store
      const int jr = x / (kD / 4), c = 4 * (x - jr * (kD / 4));
      const int owner = c / per, cl = c - owner * per;
      st_cluster_f32x4(cluster_map(rc0 + ((j * NR + jr) * per + cl) * 4, owner),
                       *reinterpret_cast<const float4 *>(stg + jr * kD + c));
    }
    if (lane < NR) {
      const float2 ml = stg_ml[lane];
#pragma unroll 1
      for (int qr = 0; qr < Q; ++qr) st_cluster_f32x2(cluster_map(ml0 + (j * NR + lane) * 8, qr), ml);
    }
    __syncwarp();
  }

  // ------------------------------------------------------------ merge
  // every partial of the cluster has been pushed and is visible; after this
  // barrier no CTA touches another's shared memory
  cluster_sync();
  {
    // CTA `rank` merges channels [rank per, (rank + 1) per) of the NR rows,
    // one thread per 4 channels of a row, from its own shared memory
    const int n4 = per / 4;
    const int Hq = H * Gc;
#pragma unroll 1
    for (int e = tid; e < NR * n4; e += kAttnThreads) {
      const int jr = e / n4, cl = 4 * (e - jr * n4);
      float M = -INFINITY;
#pragma unroll 4
      for (int jj = 0; jj < nw; ++jj) M = fmaxf(M, s_mlr[jj * NR + jr].x);
      float Ls = 0.f;
      float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int jj = 0; jj < nw; ++jj) {
        const float2 ml = s_mlr[jj * NR + jr];
        const float sc = ml.x != -INFINITY ? ex2_approx(ml.x - M) : 0.f;
        const float4 ov = *reinterpret_cast<const float4 *>(&s_recv[(jj * NR + jr) * per + cl]);
        Ls = fmaf(sc, ml.y, Ls);
        A.x = fmaf(sc, ov.x, A.x);
        A.y = fmaf(sc, ov.y, A.y);
        A.z = fmaf(sc, ov.z, A.z);
        A.w = fmaf(sc, ov.w, A.w);
      }
      const int c = rank * per + cl;
      if (Ls <= 0.f && c == 0) set_status(KVR_ST_NO_TOKENS);
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
      const int tau = CAUSAL ? jr / Gc : 0;
      const size_t row = (static_cast<size_t>(b) * T + tau) * Hq + g * Gc + jr - tau * Gc;
      const float4 r = make_float4(A.x * inv, A.y * inv, A.z * inv, A.w * inv);
      if (out_bf16)
        *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(out) + row * kD + c) =
            make_uint2(pack_bf16x2(r.x, r.y), pack_bf16x2(r.z, r.w));
      else
        *reinterpret_cast<float4 *>(static_cast<float *>(out) + row * kD + c) = r;
    }
  }
  if (early) pdl_wait();  // this grid completes after the kernel it depends on
  // every CTA of the cluster read the word at its start (all passed the
  // cluster barrier above); once the top-k has finished (the wait), nothing
  // sets it again in this call
  if (ready != nullptr && rank == 0 && tid == 0) ready[u] = 0ull;
}

}  // namespace kvr
