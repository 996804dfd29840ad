// kvr.cu -- the C ABI of libkvr (declared in include/kvr.h).
//
// Host side only: argument checks (before anything is enqueued), workspace
// carving, tensor-map encoding for the K/V pools, kernel dispatch over the
// supported (G, P) instances and the event wiring of the overlapped steps
// and of the multi-layer pipeline.  All compute is in the kernels of the
// included .cuh files.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <thread>

#include "attention.cuh"
#include "common.cuh"
#include "io.cuh"
#include "pipeline.cuh"
#include "recall.cuh"
#include "select.cuh"
#include "summaries.cuh"

namespace {

using namespace kvr;

thread_local char g_err_text[512];

// Bound of the kernels' waits for progress, passed to every streaming launch.
std::atomic<uint64_t> g_wait_limit{kWaitNs};

// Tag of one speculative step's early-start words: a per-process call count
// in the low half and a fixed pattern in the high half, so that no zeroed
// word and no earlier call's word carries it.  A CUDA graph keeps the tag of
// its capture; each replay's attention clears the words it used.
unsigned long long next_ready_tag() {
  static std::atomic<uint32_t> calls{0};
  return (0x9E3779B9ull << 32) | (calls.fetch_add(1, std::memory_order_relaxed) + 1u);
}

int cuda_fail(cudaError_t e, const char *where) {
  std::snprintf(g_err_text, sizeof g_err_text, "CUDA error in %s: %s", where,
                cudaGetErrorString(e));
  return KVR_ERR_CUDA;
}

int check_launch(const char *where) {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? KVR_OK : cuda_fail(e, where);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int check_dims(const kvr_dims *d) {
  if (!d) return KVR_ERR_INVALID_ARG;
  if (d->batch <= 0 || d->n_q_heads <= 0 || d->n_kv_heads <= 0 || d->head_dim <= 0 ||
      d->page_size <= 0 || d->n_pages <= 0 || d->n_phys_pages <= 0)
    return KVR_ERR_INVALID_ARG;
  if (d->head_dim != kD) return KVR_ERR_UNSUPPORTED_SHAPE;
  if (d->n_q_heads % d->n_kv_heads) return KVR_ERR_UNSUPPORTED_SHAPE;
  const int G = d->n_q_heads / d->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return KVR_ERR_UNSUPPORTED_SHAPE;
  if (d->page_size != 16 && d->page_size != 32 && d->page_size != 64)
    return KVR_ERR_UNSUPPORTED_SHAPE;
  if (d->n_pages > kMaxPages || d->n_kv_heads > 64 || d->batch > 65535)
    return KVR_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<int64_t>(d->n_phys_pages) * d->page_size > (int64_t{1} << 31))
    return KVR_ERR_UNSUPPORTED_SHAPE;
  return KVR_OK;
}

int check_topk(const kvr_dims *d, int32_t top_k) {
  if (top_k <= 0) return KVR_ERR_INVALID_ARG;
  if (top_k > d->n_pages) return KVR_ERR_UNSUPPORTED_SHAPE;
  return KVR_OK;
}

// Raise a kernel's dynamic shared-memory limit once per device (cached).
constexpr int kMaxDevices = 64;
int ensure_smem(const void *kern, size_t bytes, int *max_set) {
  if (bytes <= 48 * 1024) return KVR_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return KVR_ERR_UNSUPPORTED_SHAPE;
  if (max_set[dev] >= static_cast<int>(bytes)) return KVR_OK;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return cuda_fail(e, "dynamic shared memory attribute");
  // prefer the largest shared-memory carveout, so several such CTAs fit per SM
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return cuda_fail(e, "shared memory carveout attribute");
  max_set[dev] = static_cast<int>(bytes);
  return KVR_OK;
}

// Prefer the largest shared-memory carveout for a kernel with little or no
// shared memory of its own (set once per device and kernel).  An SM's split
// between L1 and shared memory follows the preferences of the kernels
// resident on it, and the attention's ring needs most of an SM's shared
// memory: the kernels that run before or beside it (top-k, the speculative
// decision, recall, append) take this preference so that an SM
// holding one of their CTAs can still take an attention CTA at once.  (Not
// the stand-in projection read: a streaming kernel of plain loads, which
// measured slower with the smaller L1.)
std::mutex g_carve_mu;
struct Carved {
  int dev;
  const void *kern;
};
Carved g_carved[256];
int g_n_carved = 0;

int prefer_max_shared(const void *kern) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_carve_mu);
  for (int i = 0; i < g_n_carved; ++i)
    if (g_carved[i].dev == dev && g_carved[i].kern == kern) return KVR_OK;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return cuda_fail(e, "shared memory carveout attribute");
  if (g_n_carved < 256) g_carved[g_n_carved++] = Carved{dev, kern};
  return KVR_OK;
}

// ---------------------------------------------------------------- workspace

struct SelectWs {
  float *scores;      // [B][H][N] fp32 page scores between the two selection kernels
  uint32_t *count;    // one word per unit, kept zero (reserved in the layout; unused)
};
struct AttnWs {
  // [B][H] words of the speculative step's early start (the attention keeps
  // its split partials on chip)
  unsigned long long *ready;
};

// Per-sequence lengths for the attention (seq_len null: every page full),
// and the several-query form: T query tokens per sequence (sel_log holds the
// logical ids of sel_phys, for the causal limits), bf16 output.
struct AttnLen {
  const int32_t *seq_len = nullptr;
  const int32_t *page_table = nullptr;
  int T = 1;
  const int32_t *sel_log = nullptr;
  int out_bf16 = 0;
  unsigned long long *ready = nullptr;  // early start of reused units (speculative step)
  unsigned long long ready_tag = 0;
};

size_t select_ws_bytes(const kvr_dims *d) {
  const size_t units = static_cast<size_t>(d->batch) * d->n_kv_heads;
  return align_up(units * d->n_pages * sizeof(float)) + align_up(units * sizeof(uint32_t));
}

size_t attn_ws_bytes(const kvr_dims *d, int top_k) {
  (void)top_k;
  const size_t units = static_cast<size_t>(d->batch) * d->n_kv_heads;
  return align_up(units * sizeof(unsigned long long));
}

// The query staged in device memory by the host-buffer step.
size_t stage_ws_bytes(const kvr_dims *d) {
  return align_up(static_cast<size_t>(d->batch) * d->n_q_heads * d->head_dim * sizeof(uint16_t));
}

SelectWs carve_select(const kvr_dims *d, uint8_t *p) {
  const size_t units = static_cast<size_t>(d->batch) * d->n_kv_heads;
  SelectWs w;
  w.scores = reinterpret_cast<float *>(p);
  w.count = reinterpret_cast<uint32_t *>(p + align_up(units * d->n_pages * sizeof(float)));
  return w;
}

AttnWs carve_attn(const kvr_dims *d, int top_k, uint8_t *p) {
  (void)d;
  (void)top_k;
  AttnWs w;
  w.ready = reinterpret_cast<unsigned long long *>(p);
  return w;
}

// ---------------------------------------------------------------- tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The pool [n_phys][P][H][D] bf16 viewed as [tokens][H][D]; one box is 64
// channels of one head over min(P, 32) consecutive token rows, written to
// shared memory with 128-byte swizzling (the attention kernel's chunk halves).
// A tensor map is a pure function of its base address, shape and box, so
// the encoded maps are kept in a small per-thread cache keyed by exactly
// those (a hit can never be stale) and eager callers skip re-encoding.
struct MapKey {
  int kind;
  const void *ptr;
  uint64_t a, b, c;
  bool operator==(const MapKey &o) const {
    return kind == o.kind && ptr == o.ptr && a == o.a && b == o.b && c == o.c;
  }
};
constexpr int kMapCache = 16;
struct MapCache {
  MapKey key[kMapCache];
  CUtensorMap map[kMapCache];
  bool valid[kMapCache] = {};
  int next = 0;
  bool find(const MapKey &k, CUtensorMap *out) const {
    for (int i = 0; i < kMapCache; ++i)
      if (valid[i] && key[i] == k) {
        *out = map[i];
        return true;
      }
    return false;
  }
  void put(const MapKey &k, const CUtensorMap &m) {
    key[next] = k;
    map[next] = m;
    valid[next] = true;
    next = (next + 1) % kMapCache;
  }
};
thread_local MapCache t_maps;

int make_pool_map(CUtensorMap *map, const void *pool, const kvr_dims *d, int64_t n_phys) {
  const MapKey key{1, pool, static_cast<uint64_t>(d->n_kv_heads), static_cast<uint64_t>(n_phys),
                   static_cast<uint64_t>(d->page_size)};
  if (t_maps.find(key, map)) return KVR_OK;
  auto fn = encode_fn();
  if (!fn) {
    std::snprintf(g_err_text, sizeof g_err_text, "cuTensorMapEncodeTiled unavailable");
    return KVR_ERR_CUDA;
  }
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(d->n_kv_heads),
                              static_cast<cuuint64_t>(n_phys * d->page_size)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2,
                                 static_cast<cuuint64_t>(d->n_kv_heads) * kD * 2};
  const cuuint32_t box[3] = {64u, 1u, static_cast<cuuint32_t>(std::min(d->page_size, 32))};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r =
      fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), dims, strides, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_err_text, sizeof g_err_text, "cuTensorMapEncodeTiled failed (%d)",
                  static_cast<int>(r));
    return KVR_ERR_CUDA;
  }
  t_maps.put(key, *map);
  return KVR_OK;
}

// The page summaries [B][H][N][2][D] bf16 viewed as [pages][256]; one box is
// 64 channels of `rows` pages, written to shared memory with 128-byte swizzling.
int make_summ_map(CUtensorMap *map, const void *summ, long long F, int rows) {
  const MapKey key{2, summ, static_cast<uint64_t>(F), static_cast<uint64_t>(rows), 0};
  if (t_maps.find(key, map)) return KVR_OK;
  auto fn = encode_fn();
  if (!fn) {
    std::snprintf(g_err_text, sizeof g_err_text, "cuTensorMapEncodeTiled unavailable");
    return KVR_ERR_CUDA;
  }
  const cuuint64_t dims[2] = {2 * static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(F)};
  const cuuint64_t strides[1] = {4 * static_cast<cuuint64_t>(kD)};
  const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r =
      fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(summ), dims, strides, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_err_text, sizeof g_err_text, "cuTensorMapEncodeTiled failed (%d)",
                  static_cast<int>(r));
    return KVR_ERR_CUDA;
  }
  t_maps.put(key, *map);
  return KVR_OK;
}

// ---------------------------------------------------------------- launches

int sm_count(int *out);

// Which kernels of the selection a launch_select call enqueues.
constexpr int kSelScores = 1;  // k_page_scores
constexpr int kSelTopk = 2;    // k_topk
constexpr int kSelBoth = kSelScores | kSelTopk;

// k_page_scores for NR = G T query rows per unit (q [B][T][Hq][D]): kScCPS
// CTAs per SM, each warp a worker over a contiguous range of the flat page
// list; a programmatic dependent launch unless pdl_first is false (right
// after an event wait): the setup overlaps the kernel before it.
template <int NR>
int launch_scores(const kvr_dims *d, const uint16_t *q, const uint16_t *summ, int T, SelectWs w,
                  float *scores, cudaStream_t st, bool pdl_first) {
  auto kern = k_page_scores<NR>;
  static int max_set[kMaxDevices] = {};
  if (int rc = ensure_smem(reinterpret_cast<const void *>(kern), kScSmem, max_set)) return rc;
  int sms = 0;
  if (int rc = sm_count(&sms)) return rc;
  const long long F = static_cast<long long>(d->batch) * d->n_kv_heads * d->n_pages;
  const long long per_cta = static_cast<long long>(kScMinPagesPerWorker) * kScNC;
  long long n_ctas = std::min<long long>(static_cast<long long>(sms) * kScCPS, (F + per_cta - 1) / per_cta);
  n_ctas = std::max<long long>(1, std::min<long long>(n_ctas, kScMaxCtas));
  CUtensorMap tsm, tsm8;
  if (int rc = make_summ_map(&tsm, summ, F, kScPages)) return rc;
  if (int rc = make_summ_map(&tsm8, summ, F, 8)) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_ctas));
  cfg.blockDim = dim3(kScThreads);
  cfg.dynamicSmemBytes = kScSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_first ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tsm, tsm8, q, d->n_kv_heads, d->n_pages, F, T,
                                           d->n_q_heads / d->n_kv_heads,
                                           g_wait_limit.load(std::memory_order_relaxed), w.scores, scores);
  if (e != cudaSuccess) return cuda_fail(e, "k_page_scores");
  return KVR_OK;
}

// T: query tokens per sequence (q [B][T][Hq][D]); more than one only
// without the speculative mode (the query rows per unit, G T, are 1, 2, 4,
// 8 or 16, checked by the callers).
template <int G>
int launch_select_g(const kvr_dims *d, const uint16_t *q, const uint16_t *summ,
                    const int32_t *ptab, int k, SelectWs w, int32_t *sel, int32_t *sel_phys,
                    float *scores, const SpecArgs &spec, cudaStream_t st, bool pdl_first,
                    const int32_t *seq_len, int parts, int T) {
  if (parts & kSelScores) {
    int rc;
    switch (G * T) {
      case 1: rc = launch_scores<1>(d, q, summ, T, w, scores, st, pdl_first); break;
      case 2: rc = launch_scores<2>(d, q, summ, T, w, scores, st, pdl_first); break;
      case 4: rc = launch_scores<4>(d, q, summ, T, w, scores, st, pdl_first); break;
      case 8: rc = launch_scores<8>(d, q, summ, T, w, scores, st, pdl_first); break;
      default: rc = launch_scores<16>(d, q, summ, T, w, scores, st, pdl_first); break;
    }
    if (rc) return rc;
  }
  if (!(parts & kSelTopk)) return KVR_OK;
  // 2. top-k per unit: a programmatic dependent launch right after the
  //    scores (an ordinary launch when it opens the stream's work after an
  //    event wait); threads x keys per thread by page count (measured: fewer
  //    than 8 keys per thread costs more in cross-warp steps than it saves)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(d->n_kv_heads, d->batch);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (parts & kSelScores) || pdl_first ? 1 : 0;
  const float *ws_sc = static_cast<const float *>(w.scores);
  cudaError_t e;
  if (d->n_pages <= 256 * 4) {
    cfg.blockDim = dim3(256);
    if (int rc = prefer_max_shared(reinterpret_cast<const void *>(k_topk<G, 256, 4>))) return rc;
    e = cudaLaunchKernelEx(&cfg, k_topk<G, 256, 4>, q, ptab, d->n_kv_heads, d->n_pages, k, ws_sc,
                           sel, sel_phys, spec, seq_len, d->page_size);
  } else if (d->n_pages <= 256 * 8) {
    cfg.blockDim = dim3(256);
    if (int rc = prefer_max_shared(reinterpret_cast<const void *>(k_topk<G, 256, 8>))) return rc;
    e = cudaLaunchKernelEx(&cfg, k_topk<G, 256, 8>, q, ptab, d->n_kv_heads, d->n_pages, k, ws_sc,
                           sel, sel_phys, spec, seq_len, d->page_size);
  } else if (d->n_pages <= 512 * 8) {
    cfg.blockDim = dim3(512);
    if (int rc = prefer_max_shared(reinterpret_cast<const void *>(k_topk<G, 512, 8>))) return rc;
    e = cudaLaunchKernelEx(&cfg, k_topk<G, 512, 8>, q, ptab, d->n_kv_heads, d->n_pages, k, ws_sc,
                           sel, sel_phys, spec, seq_len, d->page_size);
  } else if (d->n_pages <= 512 * 16) {
    cfg.blockDim = dim3(512);
    if (int rc = prefer_max_shared(reinterpret_cast<const void *>(k_topk<G, 512, 16>))) return rc;
    e = cudaLaunchKernelEx(&cfg, k_topk<G, 512, 16>, q, ptab, d->n_kv_heads, d->n_pages, k, ws_sc,
                           sel, sel_phys, spec, seq_len, d->page_size);
  } else {
    cfg.blockDim = dim3(1024);
    static_assert(1024 * 16 >= kMaxPages, "the largest top-k launch covers every page count");
    if (int rc = prefer_max_shared(reinterpret_cast<const void *>(k_topk<G, 1024, 16>))) return rc;
    e = cudaLaunchKernelEx(&cfg, k_topk<G, 1024, 16>, q, ptab, d->n_kv_heads, d->n_pages, k, ws_sc,
                           sel, sel_phys, spec, seq_len, d->page_size);
  }
  if (e != cudaSuccess) return cuda_fail(e, "k_topk");
  return KVR_OK;
}

// pdl_first: launch the scoring kernel as a programmatic dependent launch
// (false right after an event wait on the stream); seq_len (may be null):
// rank only the pages each sequence has started
int launch_select(const kvr_dims *d, const uint16_t *q, const uint16_t *summ,
                  const int32_t *ptab, int k, SelectWs w, int32_t *sel, int32_t *sel_phys,
                  float *scores, const SpecArgs &spec, cudaStream_t st, bool pdl_first = true,
                  const int32_t *seq_len = nullptr, int parts = kSelBoth, int T = 1) {
  switch (d->n_q_heads / d->n_kv_heads) {
    case 1: return launch_select_g<1>(d, q, summ, ptab, k, w, sel, sel_phys, scores, spec, st, pdl_first, seq_len, parts, T);
    case 2: return launch_select_g<2>(d, q, summ, ptab, k, w, sel, sel_phys, scores, spec, st, pdl_first, seq_len, parts, T);
    case 4: return launch_select_g<4>(d, q, summ, ptab, k, w, sel, sel_phys, scores, spec, st, pdl_first, seq_len, parts, T);
    default: return launch_select_g<8>(d, q, summ, ptab, k, w, sel, sel_phys, scores, spec, st, pdl_first, seq_len, parts, T);
  }
}

// Streaming multiprocessors of the current device (cached per device).
int sm_count(int *out) {
  static int cached[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return KVR_ERR_UNSUPPORTED_SHAPE;
  if (cached[dev] == 0) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "multiprocessor count");
    cached[dev] = n;
  }
  *out = cached[dev];
  return KVR_OK;
}

// CTAs per cluster of the attention kernel: the largest Q in {8, 4, 2} whose
// clusters for all units are resident at once (and that leaves every worker
// at least one chunk), else 1.  Occupancy per Q is cached per device.
template <int NR, int P>
int attn_cluster_size(const void *kern, size_t smem, long long units, long long kc, int *q_out) {
  static int cap[kMaxDevices][4] = {};  // resident clusters for Q = 1, 2, 4, 8 (0: not yet asked)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return KVR_ERR_UNSUPPORTED_SHAPE;
  int q = 1;
  for (int lq = 3; lq >= 1; --lq) {
    const int cand = 1 << lq;
    if (static_cast<long long>(cand) * kAttnNC > kc) continue;
    if (cap[dev][lq] == 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(cand));
      cfg.blockDim = dim3(kAttnThreads);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(cand);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess) return cuda_fail(e, "cluster occupancy");
      cap[dev][lq] = n > 0 ? n : -1;
    }
    if (cap[dev][lq] > 0 && units <= cap[dev][lq]) {
      q = cand;
      break;
    }
  }
  *q_out = q;
  return KVR_OK;
}

template <int NR, int P, bool CAUSAL>
int launch_attn_gp(const kvr_dims *d, const CUtensorMap &tk, const CUtensorMap &tv,
                   const uint16_t *q, const int32_t *sel_phys, int k, int n_phys, float scale,
                   const uint8_t *filter, int filter_mode, AttnWs w, void *out, cudaStream_t st,
                   bool pdl_ok, AttnLen len) {
  (void)w;
  using Cfg = AttnCfg<NR, P>;
  const long long units = static_cast<long long>(d->batch) * d->n_kv_heads;
  const long long kc = static_cast<long long>(k) * Cfg::CPP;
  const size_t smem = Cfg::kSmem;
  auto kern = k_sparse_decode<NR, P, CAUSAL>;
  static int max_set[kMaxDevices] = {};
  if (int rc = ensure_smem(reinterpret_cast<const void *>(kern), smem, max_set)) return rc;
  int Q = 1;
  if (int rc = attn_cluster_size<NR, P>(reinterpret_cast<const void *>(kern), smem, units, kc, &Q))
    return rc;
  if (units * Q > 0x7fffffffLL) return KVR_ERR_UNSUPPORTED_SHAPE;
  const float scale_log2 = scale * 1.4426950408889634f;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units * Q));
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  // clusters of Q CTAs, one per unit; a programmatic dependent launch (unless
  // the stream's last operation is an event wait): the setup overlaps the
  // kernel before it on the stream
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(Q);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_ok ? 2 : 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tk, tv, q, sel_phys, len.sel_log, d->n_kv_heads,
                                           k, n_phys, Q, len.T, d->n_q_heads / d->n_kv_heads,
                                           scale_log2, g_wait_limit.load(std::memory_order_relaxed),
                                           filter, filter_mode, out, len.out_bf16,
                                           len.seq_len, len.page_table, d->n_pages, len.ready,
                                           len.ready_tag);
  if (e != cudaSuccess) return cuda_fail(e, "k_sparse_decode");
  return KVR_OK;
}

template <int NR, bool CAUSAL>
int launch_attn_g(const kvr_dims *d, const CUtensorMap &tk, const CUtensorMap &tv,
                  const uint16_t *q, const int32_t *sel_phys, int k, int n_phys, float scale,
                  const uint8_t *filter, int filter_mode, AttnWs w, void *out, cudaStream_t st,
                  bool pdl_ok, AttnLen len) {
  switch (d->page_size) {
    case 16:
      return launch_attn_gp<NR, 16, CAUSAL>(d, tk, tv, q, sel_phys, k, n_phys, scale, filter,
                                            filter_mode, w, out, st, pdl_ok, len);
    case 32:
      return launch_attn_gp<NR, 32, CAUSAL>(d, tk, tv, q, sel_phys, k, n_phys, scale, filter,
                                            filter_mode, w, out, st, pdl_ok, len);
    default:
      return launch_attn_gp<NR, 64, CAUSAL>(d, tk, tv, q, sel_phys, k, n_phys, scale, filter,
                                            filter_mode, w, out, st, pdl_ok, len);
  }
}

// pdl_ok: launch as a programmatic dependent launch (false right after an
// event wait on the stream, whose dependency must stay a full one).  The
// query rows per unit, G len.T, are 1, 2, 4, 8 or 16 (checked by the callers).
int launch_attn(const kvr_dims *d, const uint16_t *q, const uint16_t *k_pool,
                const uint16_t *v_pool, int64_t n_phys, const int32_t *sel_phys, int k,
                float scale, const uint8_t *filter, int filter_mode, AttnWs w, void *out,
                cudaStream_t st, bool pdl_ok = true, AttnLen len = AttnLen()) {
  CUtensorMap tk, tv;
  int rc = make_pool_map(&tk, k_pool, d, n_phys);
  if (rc) return rc;
  rc = make_pool_map(&tv, v_pool, d, n_phys);
  if (rc) return rc;
  if (!(scale > 0.f)) scale = 1.0f / std::sqrt(static_cast<float>(kD));
  const int np = static_cast<int>(n_phys);
  if (len.T == 1) {  // one query token: no causal limits (G <= 8 rows)
    switch (d->n_q_heads / d->n_kv_heads) {
      case 1: return launch_attn_g<1, false>(d, tk, tv, q, sel_phys, k, np, scale, filter, filter_mode, w, out, st, pdl_ok, len);
      case 2: return launch_attn_g<2, false>(d, tk, tv, q, sel_phys, k, np, scale, filter, filter_mode, w, out, st, pdl_ok, len);
      case 4: return launch_attn_g<4, false>(d, tk, tv, q, sel_phys, k, np, scale, filter, filter_mode, w, out, st, pdl_ok, len);
      default: return launch_attn_g<8, false>(d, tk, tv, q, sel_phys, k, np, scale, filter, filter_mode, w, out, st, pdl_ok, len);
    }
  }
  switch (d->n_q_heads / d->n_kv_heads * len.T) {
    case 2: return launch_attn_g<2, true>(d, tk, tv, q, sel_phys, k, np, scale, filter, filter_mode, w, out, st, pdl_ok, len);
    case 4: return launch_attn_g<4, true>(d, tk, tv, q, sel_phys, k, np, scale, filter, filter_mode, w, out, st, pdl_ok, len);
    case 8: return launch_attn_g<8, true>(d, tk, tv, q, sel_phys, k, np, scale, filter, filter_mode, w, out, st, pdl_ok, len);
    default: return launch_attn_g<16, true>(d, tk, tv, q, sel_phys, k, np, scale, filter, filter_mode, w, out, st, pdl_ok, len);
  }
}

// Device address of page-locked host memory (the kernels read or write it
// directly); `what` names the buffer in the error text.
int mapped_host_pointer(const void *host, void **dev, const char *what = "host cache") {
  cudaPointerAttributes a;
  const cudaError_t e = cudaPointerGetAttributes(&a, host);
  if (e != cudaSuccess) return cuda_fail(e, what);
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) {
    std::snprintf(g_err_text, sizeof g_err_text, "%s is not page-locked, mapped host memory", what);
    return KVR_ERR_INVALID_ARG;
  }
  *dev = a.devicePointer;
  return KVR_OK;
}

int launch_recall(const kvr_dims *d, const kvr_host_kv *host, const kvr_working_set *wset,
                  const int32_t *sel_new, const int32_t *protect, const uint8_t *corrected,
                  int k, int32_t *sel_slot_out, uint32_t *n_copied, cudaStream_t st,
                  int unit_filter = 0) {
  void *kh = nullptr, *vh = nullptr;
  int rc = mapped_host_pointer(host->k_host, &kh);
  if (rc) return rc;
  if ((rc = mapped_host_pointer(host->v_host, &vh))) return rc;
  const int S = wset->n_slots;
  const size_t smem = (2 * static_cast<size_t>(S) + k) * sizeof(int32_t);
  const dim3 grid(d->n_kv_heads, d->batch);
#define KVR_RECALL(PP)                                                                          \
  if (int rc2 = prefer_max_shared(reinterpret_cast<const void *>(k_recall<PP>))) return rc2;   \
  k_recall<PP><<<grid, kRecallThreads, smem, st>>>(                                             \
      static_cast<const uint16_t *>(kh), static_cast<const uint16_t *>(vh), wset->k_slots,      \
      wset->v_slots, wset->page2slot, wset->slot2page, S, sel_new, protect, corrected,          \
      unit_filter, d->n_kv_heads, d->n_pages, k, sel_slot_out, n_copied)
  switch (d->page_size) {
    case 16: KVR_RECALL(16); break;
    case 32: KVR_RECALL(32); break;
    default: KVR_RECALL(64); break;
  }
#undef KVR_RECALL
  return check_launch("k_recall");
}

int check_wset(const kvr_dims *d, const kvr_working_set *w, int32_t top_k) {
  if (!w || !w->k_slots || !w->v_slots || !w->page2slot || !w->slot2page) return KVR_ERR_INVALID_ARG;
  if (w->n_slots < 2 * top_k) return KVR_ERR_UNSUPPORTED_SHAPE;
  if ((2 * static_cast<int64_t>(w->n_slots) + top_k) * 4 > 48 * 1024) return KVR_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<int64_t>(d->batch) * w->n_slots * d->page_size > (int64_t{1} << 31))
    return KVR_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(w->k_slots) || !aligned16(w->v_slots) || !aligned16(w->page2slot) ||
      !aligned16(w->slot2page))
    return KVR_ERR_ALIGN;
  return KVR_OK;
}

int check_ws(void *ws, size_t have, size_t need) {
  if (!ws) return KVR_ERR_WORKSPACE;
  if (have < need) return KVR_ERR_WORKSPACE;
  if (!aligned16(ws)) return KVR_ERR_ALIGN;
  return KVR_OK;
}

SpecArgs no_spec() {
  SpecArgs s;
  std::memset(&s, 0, sizeof s);
  return s;
}

template <int G>
int launch_spec_decide_g(const kvr_dims *d, const uint16_t *q, const int32_t *ptab, int k,
                         const SpecArgs &spec, cudaStream_t st) {
  if (int rc = prefer_max_shared(reinterpret_cast<const void *>(k_spec_decide<G>))) return rc;
  k_spec_decide<G><<<dim3(d->n_kv_heads, d->batch), 32 * G, 0, st>>>(q, ptab, d->n_kv_heads,
                                                                     d->n_pages, k, spec);
  return check_launch("k_spec_decide");
}

int launch_spec_decide(const kvr_dims *d, const uint16_t *q, const int32_t *ptab, int k,
                       const SpecArgs &spec, cudaStream_t st) {
  switch (d->n_q_heads / d->n_kv_heads) {
    case 1: return launch_spec_decide_g<1>(d, q, ptab, k, spec, st);
    case 2: return launch_spec_decide_g<2>(d, q, ptab, k, spec, st);
    case 4: return launch_spec_decide_g<4>(d, q, ptab, k, spec, st);
    default: return launch_spec_decide_g<8>(d, q, ptab, k, spec, st);
  }
}

}  // namespace

extern "C" {

size_t kvr_workspace_size(const kvr_dims *dims, int32_t top_k, int32_t op) {
  if (check_dims(dims) || check_topk(dims, top_k)) return 0;
  switch (op) {
    case KVR_OP_SELECT: return select_ws_bytes(dims);
    case KVR_OP_ATTN: return attn_ws_bytes(dims, top_k);
    case KVR_OP_STEP: return select_ws_bytes(dims) + attn_ws_bytes(dims, top_k);
    case KVR_OP_STEP_HOST:
      return select_ws_bytes(dims) + attn_ws_bytes(dims, top_k) + stage_ws_bytes(dims);
    default: return 0;
  }
}

static int build_summaries_impl(const kvr_dims *dims, const uint16_t *k_pool,
                                const int32_t *page_table, const int32_t *seq_len,
                                uint16_t *summ, void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!k_pool || !page_table || !summ) return KVR_ERR_INVALID_ARG;
  if (!aligned16(k_pool) || !aligned16(page_table) || !aligned16(summ) ||
      (seq_len && !aligned16(seq_len)))
    return KVR_ERR_ALIGN;
  const int cols = dims->n_kv_heads * 16;
  const int ppc = cols >= kSumThreads ? 1 : kSumThreads / cols;
  const dim3 grid((dims->n_pages + ppc - 1) / ppc, dims->batch);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (dims->page_size) {
    case 16:
      k_build_summaries<16><<<grid, kSumThreads, 0, st>>>(k_pool, page_table, seq_len, summ,
                                                          dims->n_kv_heads, dims->n_pages,
                                                          dims->n_phys_pages, ppc);
      break;
    case 32:
      k_build_summaries<32><<<grid, kSumThreads, 0, st>>>(k_pool, page_table, seq_len, summ,
                                                          dims->n_kv_heads, dims->n_pages,
                                                          dims->n_phys_pages, ppc);
      break;
    default:
      k_build_summaries<64><<<grid, kSumThreads, 0, st>>>(k_pool, page_table, seq_len, summ,
                                                          dims->n_kv_heads, dims->n_pages,
                                                          dims->n_phys_pages, ppc);
      break;
  }
  return check_launch("k_build_summaries");
}

int kvr_build_summaries(const kvr_dims *dims, const uint16_t *k_pool, const int32_t *page_table,
                        uint16_t *summ, void *stream) {
  return build_summaries_impl(dims, k_pool, page_table, nullptr, summ, stream);
}

int kvr_build_summaries_len(const kvr_dims *dims, const uint16_t *k_pool,
                            const int32_t *page_table, const int32_t *seq_len, uint16_t *summ,
                            void *stream) {
  if (!seq_len) return KVR_ERR_INVALID_ARG;
  return build_summaries_impl(dims, k_pool, page_table, seq_len, summ, stream);
}

int kvr_append_kv(const kvr_dims *dims, const uint16_t *k_new, const uint16_t *v_new,
                  const int32_t *page_table, int32_t *seq_len, uint16_t *k_pool,
                  uint16_t *v_pool, uint16_t *summ, void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!k_new || !v_new || !page_table || !seq_len || !k_pool || !v_pool || !summ)
    return KVR_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(page_table) || !aligned16(seq_len) ||
      !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(summ))
    return KVR_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dim3 grid(dims->batch);
#define KVR_APPEND(PP)                                                                        \
  if ((rc = prefer_max_shared(reinterpret_cast<const void *>(k_append<PP>)))) return rc;       \
  k_append<PP><<<grid, kAppendThreads, 0, st>>>(k_new, v_new, page_table, seq_len, k_pool,    \
                                                v_pool, summ, dims->n_kv_heads, dims->n_pages, \
                                                dims->n_phys_pages)
  switch (dims->page_size) {
    case 16: KVR_APPEND(16); break;
    case 32: KVR_APPEND(32); break;
    default: KVR_APPEND(64); break;
  }
#undef KVR_APPEND
  return check_launch("k_append");
}

int kvr_select_pages(const kvr_dims *dims, const uint16_t *q, const uint16_t *summ,
                     const int32_t *page_table, int32_t top_k, int32_t *sel, int32_t *sel_phys,
                     float *scores_opt, void *ws, size_t ws_bytes, void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_topk(dims, top_k))) return rc;
  if (!q || !summ || !page_table || !sel) return KVR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(summ) || !aligned16(page_table) || !aligned16(sel) ||
      (sel_phys && !aligned16(sel_phys)) || (scores_opt && !aligned16(scores_opt)))
    return KVR_ERR_ALIGN;
  if ((rc = check_ws(ws, ws_bytes, select_ws_bytes(dims)))) return rc;
  return launch_select(dims, q, summ, page_table, top_k, carve_select(dims, (uint8_t *)ws), sel,
                       sel_phys, scores_opt, no_spec(), static_cast<cudaStream_t>(stream));
}

int kvr_sparse_decode_attn(const kvr_dims *dims, const uint16_t *q, const uint16_t *k_pool,
                           const uint16_t *v_pool, const int32_t *sel_phys, int32_t top_k,
                           float scale, float *out, void *ws, size_t ws_bytes, void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_topk(dims, top_k))) return rc;
  if (!q || !k_pool || !v_pool || !sel_phys || !out) return KVR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(sel_phys) ||
      !aligned16(out))
    return KVR_ERR_ALIGN;
  if (std::isnan(scale)) return KVR_ERR_INVALID_ARG;
  if ((rc = check_ws(ws, ws_bytes, attn_ws_bytes(dims, top_k)))) return rc;
  return launch_attn(dims, q, k_pool, v_pool, dims->n_phys_pages, sel_phys, top_k, scale, nullptr,
                     0, carve_attn(dims, top_k, (uint8_t *)ws), out,
                     static_cast<cudaStream_t>(stream));
}

int kvr_select_pages_len(const kvr_dims *dims, const uint16_t *q, const uint16_t *summ,
                         const int32_t *page_table, const int32_t *seq_len, int32_t top_k,
                         int32_t *sel, int32_t *sel_phys, float *scores_opt, void *ws,
                         size_t ws_bytes, void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_topk(dims, top_k))) return rc;
  if (!q || !summ || !page_table || !seq_len || !sel) return KVR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(summ) || !aligned16(page_table) || !aligned16(seq_len) ||
      !aligned16(sel) || (sel_phys && !aligned16(sel_phys)) ||
      (scores_opt && !aligned16(scores_opt)))
    return KVR_ERR_ALIGN;
  if ((rc = check_ws(ws, ws_bytes, select_ws_bytes(dims)))) return rc;
  return launch_select(dims, q, summ, page_table, top_k, carve_select(dims, (uint8_t *)ws), sel,
                       sel_phys, scores_opt, no_spec(), static_cast<cudaStream_t>(stream), true,
                       seq_len);
}

int kvr_sparse_decode_attn_len(const kvr_dims *dims, const uint16_t *q, const uint16_t *k_pool,
                               const uint16_t *v_pool, const int32_t *page_table,
                               const int32_t *seq_len, const int32_t *sel_phys, int32_t top_k,
                               float scale, float *out, void *ws, size_t ws_bytes,
                               void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_topk(dims, top_k))) return rc;
  if (!q || !k_pool || !v_pool || !page_table || !seq_len || !sel_phys || !out)
    return KVR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(page_table) ||
      !aligned16(seq_len) || !aligned16(sel_phys) || !aligned16(out))
    return KVR_ERR_ALIGN;
  if (std::isnan(scale)) return KVR_ERR_INVALID_ARG;
  if ((rc = check_ws(ws, ws_bytes, attn_ws_bytes(dims, top_k)))) return rc;
  AttnLen len;
  len.seq_len = seq_len;
  len.page_table = page_table;
  return launch_attn(dims, q, k_pool, v_pool, dims->n_phys_pages, sel_phys, top_k, scale, nullptr,
                     0, carve_attn(dims, top_k, (uint8_t *)ws), out,
                     static_cast<cudaStream_t>(stream), true, len);
}

// Query rows per unit of a several-queries call: G T in {1, 2, 4, 8, 16}.
static int check_rows(const kvr_dims *dims, int32_t n_query) {
  if (n_query <= 0) return KVR_ERR_INVALID_ARG;
  const int64_t nr = static_cast<int64_t>(dims->n_q_heads / dims->n_kv_heads) * n_query;
  if (nr != 1 && nr != 2 && nr != 4 && nr != 8 && nr != 16) return KVR_ERR_UNSUPPORTED_SHAPE;
  return KVR_OK;
}

int kvr_select_pages_multi(const kvr_dims *dims, const uint16_t *qs, int32_t n_query,
                           const uint16_t *summ, const int32_t *page_table, const int32_t *seq_len,
                           int32_t top_k, int32_t *sel, int32_t *sel_phys, float *scores_opt,
                           void *ws, size_t ws_bytes, void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_topk(dims, top_k))) return rc;
  if ((rc = check_rows(dims, n_query))) return rc;
  if (!qs || !summ || !page_table || !seq_len || !sel) return KVR_ERR_INVALID_ARG;
  if (!aligned16(qs) || !aligned16(summ) || !aligned16(page_table) || !aligned16(seq_len) ||
      !aligned16(sel) || (sel_phys && !aligned16(sel_phys)) || (scores_opt && !aligned16(scores_opt)))
    return KVR_ERR_ALIGN;
  if ((rc = check_ws(ws, ws_bytes, select_ws_bytes(dims)))) return rc;
  return launch_select(dims, qs, summ, page_table, top_k, carve_select(dims, (uint8_t *)ws), sel,
                       sel_phys, scores_opt, no_spec(), static_cast<cudaStream_t>(stream), true,
                       seq_len, kSelBoth, n_query);
}

int kvr_sparse_decode_attn_multi(const kvr_dims *dims, const uint16_t *qs, int32_t n_query,
                                 const uint16_t *k_pool, const uint16_t *v_pool,
                                 const int32_t *page_table, const int32_t *seq_len,
                                 const int32_t *sel, const int32_t *sel_phys, int32_t top_k,
                                 float scale, void *out, int32_t out_dtype, void *ws,
                                 size_t ws_bytes, void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_topk(dims, top_k))) return rc;
  if ((rc = check_rows(dims, n_query))) return rc;
  if (out_dtype != KVR_DTYPE_F32 && out_dtype != KVR_DTYPE_BF16) return KVR_ERR_INVALID_ARG;
  if (!qs || !k_pool || !v_pool || !page_table || !seq_len || !sel_phys || !out) return KVR_ERR_INVALID_ARG;
  if (n_query > 1 && !sel) return KVR_ERR_INVALID_ARG;
  if (!aligned16(qs) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(page_table) ||
      !aligned16(seq_len) || !aligned16(sel_phys) || (sel && !aligned16(sel)) || !aligned16(out))
    return KVR_ERR_ALIGN;
  if (std::isnan(scale)) return KVR_ERR_INVALID_ARG;
  if ((rc = check_ws(ws, ws_bytes, attn_ws_bytes(dims, top_k)))) return rc;
  AttnLen len;
  len.seq_len = seq_len;
  len.page_table = page_table;
  len.T = n_query;
  len.sel_log = n_query > 1 ? sel : nullptr;
  len.out_bf16 = out_dtype == KVR_DTYPE_BF16 ? 1 : 0;
  return launch_attn(dims, qs, k_pool, v_pool, dims->n_phys_pages, sel_phys, top_k, scale, nullptr,
                     0, carve_attn(dims, top_k, (uint8_t *)ws), out,
                     static_cast<cudaStream_t>(stream), true, len);
}

static SpecArgs spec_args(const kvr_spec_state *st, float tau, uint8_t *corrected,
                          float *cbar_opt, int32_t *sel_used, int32_t *sel_used_phys,
                          const int32_t *page2slot, int n_slots) {
  SpecArgs s = no_spec();
  s.enabled = 1;
  s.step = st->step;
  s.tau = tau;
  s.q_prev = st->q_prev;
  s.sel_prev = st->sel_prev;
  s.corrected = corrected;
  s.cbar = cbar_opt;
  s.sel_used = sel_used;
  s.sel_used_phys = sel_used_phys;
  s.page2slot = page2slot;
  s.n_slots = n_slots;
  return s;
}

static int spec_select_impl(const kvr_dims *dims, kvr_spec_state *st, const uint16_t *q_t,
                            const uint16_t *summ, const int32_t *page_table, int32_t top_k,
                            float tau, uint8_t *corrected, float *cbar_opt, int32_t *sel_used,
                            int32_t *sel_used_phys, const int32_t *page2slot, int n_slots,
                            void *ws, cudaStream_t stream, bool pdl_first = true,
                            unsigned long long *ready = nullptr, unsigned long long ready_tag = 0) {
  SpecArgs s = spec_args(st, tau, corrected, cbar_opt, sel_used, sel_used_phys, page2slot, n_slots);
  s.ready = ready;
  s.ready_tag = ready_tag;
  return launch_select(dims, q_t, summ, page_table, top_k, carve_select(dims, (uint8_t *)ws),
                       nullptr, nullptr, nullptr, s, stream, pdl_first);
}

static int check_spec(const kvr_dims *dims, const kvr_spec_state *st, const uint16_t *q_t,
                      const uint16_t *summ, uint8_t *corrected, float *cbar_opt,
                      int32_t *sel_used, float tau) {
  if (!st || !st->q_prev || !st->sel_prev || st->step < 0) return KVR_ERR_INVALID_ARG;
  if (!q_t || !summ || !corrected || !sel_used) return KVR_ERR_INVALID_ARG;
  if (std::isnan(tau)) return KVR_ERR_INVALID_ARG;
  if (!aligned16(st->q_prev) || !aligned16(st->sel_prev) || !aligned16(q_t) || !aligned16(summ) ||
      !aligned16(sel_used) || (cbar_opt && !aligned16(cbar_opt)))
    return KVR_ERR_ALIGN;
  (void)dims;
  return KVR_OK;
}

int kvr_speculative_select(const kvr_dims *dims, kvr_spec_state *st, const uint16_t *q_t,
                           const uint16_t *summ, const int32_t *page_table, int32_t top_k,
                           float tau, uint8_t *corrected, float *cbar_opt, int32_t *sel_used,
                           int32_t *sel_used_phys, void *ws, size_t ws_bytes, void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_topk(dims, top_k))) return rc;
  if ((rc = check_spec(dims, st, q_t, summ, corrected, cbar_opt, sel_used, tau))) return rc;
  if (!page_table) return KVR_ERR_INVALID_ARG;
  if (!aligned16(page_table) || (sel_used_phys && !aligned16(sel_used_phys))) return KVR_ERR_ALIGN;
  if ((rc = check_ws(ws, ws_bytes, select_ws_bytes(dims)))) return rc;
  rc = spec_select_impl(dims, st, q_t, summ, page_table, top_k, tau, corrected, cbar_opt, sel_used,
                        sel_used_phys, nullptr, 0, ws, static_cast<cudaStream_t>(stream));
  if (rc == KVR_OK) st->step += 1;
  return rc;
}

int kvr_speculative_step(const kvr_dims *dims, kvr_spec_state *st, const uint16_t *q_t,
                         const uint16_t *summ, const int32_t *page_table, const uint16_t *k_pool,
                         const uint16_t *v_pool, int32_t top_k, float tau, float scale,
                         float *out, uint8_t *corrected, float *cbar_opt, int32_t *sel_used,
                         int32_t *sel_used_phys, void *ws, size_t ws_bytes, void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_topk(dims, top_k))) return rc;
  if ((rc = check_spec(dims, st, q_t, summ, corrected, cbar_opt, sel_used, tau))) return rc;
  if (!page_table || !k_pool || !v_pool || !out || !sel_used_phys) return KVR_ERR_INVALID_ARG;
  if (!aligned16(page_table) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) ||
      !aligned16(sel_used_phys))
    return KVR_ERR_ALIGN;
  if (std::isnan(scale)) return KVR_ERR_INVALID_ARG;
  if ((rc = check_ws(ws, ws_bytes, select_ws_bytes(dims) + attn_ws_bytes(dims, top_k)))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the attention of a reused unit starts as soon as the top-k's prologue
  // has announced its page ids
  const AttnWs aw = carve_attn(dims, top_k, (uint8_t *)ws + select_ws_bytes(dims));
  AttnLen early;
  early.ready = aw.ready;
  early.ready_tag = next_ready_tag();
  rc = spec_select_impl(dims, st, q_t, summ, page_table, top_k, tau, corrected, cbar_opt, sel_used,
                        sel_used_phys, nullptr, 0, ws, s, true, early.ready, early.ready_tag);
  if (rc) return rc;
  st->step += 1;
  return launch_attn(dims, q_t, k_pool, v_pool, dims->n_phys_pages, sel_used_phys, top_k, scale,
                     nullptr, 0, aw, out, s, true, early);
}

int kvr_speculative_step_host(const kvr_dims *dims, kvr_spec_state *st, const uint16_t *q_host,
                              const uint16_t *summ, const int32_t *page_table, const uint16_t *k_pool,
                              const uint16_t *v_pool, int32_t top_k, float tau, float scale,
                              float *out_host, uint8_t *corrected, float *cbar_opt, int32_t *sel_used,
                              int32_t *sel_used_phys, void *ws, size_t ws_bytes, void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_topk(dims, top_k))) return rc;
  if (!q_host || !out_host) return KVR_ERR_INVALID_ARG;
  const size_t sel_b = select_ws_bytes(dims), attn_b = attn_ws_bytes(dims, top_k);
  if ((rc = check_ws(ws, ws_bytes, sel_b + attn_b + stage_ws_bytes(dims)))) return rc;
  uint16_t *q_stage = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws) + sel_b + attn_b);
  if ((rc = check_spec(dims, st, q_stage, summ, corrected, cbar_opt, sel_used, tau))) return rc;
  if (!page_table || !k_pool || !v_pool || !sel_used_phys) return KVR_ERR_INVALID_ARG;
  if (!aligned16(page_table) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(sel_used_phys))
    return KVR_ERR_ALIGN;
  if (std::isnan(scale)) return KVR_ERR_INVALID_ARG;
  void *q_dev = nullptr, *out_dev = nullptr;
  if ((rc = mapped_host_pointer(q_host, &q_dev, "q_host"))) return rc;
  if ((rc = mapped_host_pointer(out_host, &out_dev, "out_host"))) return rc;
  if (!aligned16(q_dev) || !aligned16(out_dev)) return KVR_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint64_t n16 = static_cast<uint64_t>(dims->batch) * dims->n_q_heads * dims->head_dim * 2 / 16;
  int sms = 0;
  if ((rc = sm_count(&sms))) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(
      std::max<uint64_t>(1, std::min<uint64_t>((n16 + kStageThreads - 1) / kStageThreads, 4ull * sms))));
  cfg.blockDim = dim3(kStageThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k_stage_in, static_cast<const uint4 *>(q_dev),
                                           reinterpret_cast<uint4 *>(q_stage), n16);
  if (e != cudaSuccess) return cuda_fail(e, "k_stage_in");
  const AttnWs aw = carve_attn(dims, top_k, static_cast<uint8_t *>(ws) + sel_b);
  AttnLen early;
  early.ready = aw.ready;
  early.ready_tag = next_ready_tag();
  rc = spec_select_impl(dims, st, q_stage, summ, page_table, top_k, tau, corrected, cbar_opt, sel_used,
                        sel_used_phys, nullptr, 0, ws, s, true, early.ready, early.ready_tag);
  if (rc) return rc;
  st->step += 1;
  return launch_attn(dims, q_stage, k_pool, v_pool, dims->n_phys_pages, sel_used_phys, top_k, scale,
                     nullptr, 0, aw, out_dev, s, true, early);
}

int kvr_speculative_step_overlap(const kvr_dims *dims, kvr_spec_state *st, const uint16_t *q_t,
                                 const uint16_t *summ, const int32_t *page_table,
                                 const uint16_t *k_pool, const uint16_t *v_pool, int32_t top_k,
                                 float tau, float scale, float *out, uint8_t *corrected,
                                 float *cbar_opt, int32_t *sel_used, int32_t *sel_used_phys,
                                 void *ws, size_t ws_bytes, void *stream, void *side_stream,
                                 void *ev_decide, void *ev_select) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_topk(dims, top_k))) return rc;
  if ((rc = check_spec(dims, st, q_t, summ, corrected, cbar_opt, sel_used, tau))) return rc;
  if (!page_table || !k_pool || !v_pool || !out || !sel_used_phys || !ev_decide || !ev_select)
    return KVR_ERR_INVALID_ARG;
  if (!aligned16(page_table) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) ||
      !aligned16(sel_used_phys))
    return KVR_ERR_ALIGN;
  if (std::isnan(scale)) return KVR_ERR_INVALID_ARG;
  if ((rc = check_ws(ws, ws_bytes, select_ws_bytes(dims) + attn_ws_bytes(dims, top_k)))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t side = static_cast<cudaStream_t>(side_stream);
  cudaEvent_t ed = static_cast<cudaEvent_t>(ev_decide), es = static_cast<cudaEvent_t>(ev_select);
  SpecArgs sa = spec_args(st, tau, corrected, cbar_opt, sel_used, sel_used_phys, nullptr, 0);
  const SelectWs sw = carve_select(dims, (uint8_t *)ws);
  // 1. the decision per (b, g) (reused heads get sel_used from sel_prev),
  //    then the page scores, both on `stream`
  rc = launch_spec_decide(dims, q_t, page_table, top_k, sa, s);
  if (rc) return rc;
  st->step += 1;
  sa.decided = 1;
  rc = launch_select(dims, q_t, summ, page_table, top_k, sw, nullptr, nullptr, nullptr, sa, s, true,
                     nullptr, kSelScores);
  if (rc) return rc;
  cudaError_t e = cudaEventRecord(ed, s);
  if (e != cudaSuccess) return cuda_fail(e, "record decide event");
  // 2. side stream: the top-k of the new selection (becomes sel_prev; sel_used
  //    of the corrected heads), beside the reused heads' attention
  e = cudaStreamWaitEvent(side, ed, 0);
  if (e != cudaSuccess) return cuda_fail(e, "side stream wait");
  rc = launch_select(dims, q_t, summ, page_table, top_k, sw, nullptr, nullptr, nullptr, sa, side, false,
                     nullptr, kSelTopk);
  if (rc) return rc;
  e = cudaEventRecord(es, side);
  if (e != cudaSuccess) return cuda_fail(e, "record select event");
  // 3. attention: the reused heads alongside the selection, the corrected
  //    heads once it is done
  const AttnWs aw = carve_attn(dims, top_k, (uint8_t *)ws + select_ws_bytes(dims));
  rc = launch_attn(dims, q_t, k_pool, v_pool, dims->n_phys_pages, sel_used_phys, top_k, scale,
                   corrected, 1, aw, out, s);
  if (rc) return rc;
  e = cudaStreamWaitEvent(s, es, 0);
  if (e != cudaSuccess) return cuda_fail(e, "main stream wait");
  return launch_attn(dims, q_t, k_pool, v_pool, dims->n_phys_pages, sel_used_phys, top_k, scale,
                     corrected, 2, aw, out, s, false);
}

int kvr_working_set_reset(const kvr_dims *dims, const kvr_working_set *wset, void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!wset || !wset->page2slot || !wset->slot2page || wset->n_slots <= 0) return KVR_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t units = static_cast<size_t>(dims->batch) * dims->n_kv_heads;
  cudaError_t e = cudaMemsetAsync(wset->page2slot, 0xff, units * dims->n_pages * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(wset->slot2page, 0xff, units * wset->n_slots * 4, s);
  return e == cudaSuccess ? KVR_OK : cuda_fail(e, "working set reset");
}

int kvr_recall_pages(const kvr_dims *dims, const kvr_host_kv *host, const kvr_working_set *wset,
                     const int32_t *sel_new, const int32_t *protect, const uint8_t *corrected,
                     int32_t top_k, int32_t *sel_slot_out, uint32_t *n_copied_opt, void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_topk(dims, top_k))) return rc;
  if ((rc = check_wset(dims, wset, top_k))) return rc;
  if (!host || !host->k_host || !host->v_host || !sel_new || !protect) return KVR_ERR_INVALID_ARG;
  if (corrected && !sel_slot_out) return KVR_ERR_INVALID_ARG;
  if (!aligned16(host->k_host) || !aligned16(host->v_host) || !aligned16(sel_new) ||
      !aligned16(protect) || (sel_slot_out && !aligned16(sel_slot_out)))
    return KVR_ERR_ALIGN;
  return launch_recall(dims, host, wset, sel_new, protect, corrected, top_k, sel_slot_out,
                       n_copied_opt, static_cast<cudaStream_t>(stream));
}

int kvr_speculative_step_recall(const kvr_dims *dims, kvr_spec_state *st, const uint16_t *q_t,
                                const uint16_t *summ, const kvr_host_kv *host,
                                const kvr_working_set *wset, int32_t top_k, float tau,
                                float scale, float *out, uint8_t *corrected, float *cbar_opt,
                                int32_t *sel_used, int32_t *sel_used_slot,
                                uint32_t *n_copied_opt, void *ws, size_t ws_bytes, void *stream,
                                void *side_stream, void *ev_select, void *ev_recall) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_topk(dims, top_k))) return rc;
  if ((rc = check_spec(dims, st, q_t, summ, corrected, cbar_opt, sel_used, tau))) return rc;
  if ((rc = check_wset(dims, wset, top_k))) return rc;
  if (!host || !host->k_host || !host->v_host || !out || !sel_used_slot || !ev_select ||
      !ev_recall)
    return KVR_ERR_INVALID_ARG;
  if (!aligned16(host->k_host) || !aligned16(host->v_host) || !aligned16(out) ||
      !aligned16(sel_used_slot))
    return KVR_ERR_ALIGN;
  if (std::isnan(scale)) return KVR_ERR_INVALID_ARG;
  if ((rc = check_ws(ws, ws_bytes, select_ws_bytes(dims) + attn_ws_bytes(dims, top_k)))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t side = static_cast<cudaStream_t>(side_stream);
  cudaEvent_t es = static_cast<cudaEvent_t>(ev_select), er = static_cast<cudaEvent_t>(ev_recall);

  // 1. selection; reused heads get their (resident) slots from page2slot
  rc = spec_select_impl(dims, st, q_t, summ, nullptr, top_k, tau,
                        corrected, cbar_opt, sel_used, sel_used_slot, wset->page2slot,
                        wset->n_slots, ws, s);
  if (rc) return rc;
  st->step += 1;
  cudaError_t e = cudaEventRecord(es, s);
  if (e != cudaSuccess) return cuda_fail(e, "record select event");
  // 2. side stream: recall the new selection (now in sel_prev), protecting sel_used
  e = cudaStreamWaitEvent(side, es, 0);
  if (e != cudaSuccess) return cuda_fail(e, "side stream wait");
  rc = launch_recall(dims, host, wset, st->sel_prev, sel_used, corrected, top_k, sel_used_slot,
                     n_copied_opt, side);
  if (rc) return rc;
  e = cudaEventRecord(er, side);
  if (e != cudaSuccess) return cuda_fail(e, "record recall event");
  // 3. attention: reused heads now, corrected heads once their pages are in
  const int64_t n_phys = static_cast<int64_t>(dims->batch) * wset->n_slots;
  const AttnWs aw = carve_attn(dims, top_k, (uint8_t *)ws + select_ws_bytes(dims));
  rc = launch_attn(dims, q_t, wset->k_slots, wset->v_slots, n_phys, sel_used_slot, top_k, scale,
                   corrected, 1, aw, out, s, false);
  if (rc) return rc;
  e = cudaStreamWaitEvent(s, er, 0);
  if (e != cudaSuccess) return cuda_fail(e, "main stream wait");
  return launch_attn(dims, q_t, wset->k_slots, wset->v_slots, n_phys, sel_used_slot, top_k, scale,
                     corrected, 2, aw, out, s, false);
}

// ---------------------------------------------------------------- multi-layer pipeline

// The stand-in for a projection: k_stand_in over `bytes` of the weights from
// `offset` (nothing for bytes == 0 or no stand-in).
static int launch_stand_in(const kvr_stand_in *c, uint64_t offset, uint64_t bytes,
                           cudaStream_t st) {
  if (!c || bytes == 0) return KVR_OK;
  int sms = 0;
  if (int rc = sm_count(&sms)) return rc;
  const uint64_t n16 = bytes / 16;
  const uint64_t want = (n16 + kStandInThreads - 1) / kStandInThreads;
  const uint64_t cap = static_cast<uint64_t>(sms) * kStandInCPS;
  const unsigned grid = static_cast<unsigned>(std::max<uint64_t>(1, std::min(want, cap)));
  const uint8_t *base = static_cast<const uint8_t *>(c->weights) + offset;
  k_stand_in<<<grid, kStandInThreads, 0, st>>>(reinterpret_cast<const uint4 *>(base), n16, c->sink);
  return check_launch("k_stand_in");
}

static int check_stand_in(const kvr_stand_in *c) {
  if (!c->weights || !c->sink) return KVR_ERR_INVALID_ARG;
  if ((c->qkv_bytes | c->post_bytes) & 15u) return KVR_ERR_INVALID_ARG;
  if (c->qkv_bytes > UINT64_MAX - c->post_bytes) return KVR_ERR_INVALID_ARG;
  if (!aligned16(c->weights) || (reinterpret_cast<uintptr_t>(c->sink) & 3u)) return KVR_ERR_ALIGN;
  return KVR_OK;
}

int kvr_stand_in_read(const kvr_stand_in *compute, uint64_t offset, uint64_t bytes, void *stream) {
  if (!compute) return KVR_ERR_INVALID_ARG;
  int rc = check_stand_in(compute);
  if (rc) return rc;
  if ((offset | bytes) & 15u || offset > UINT64_MAX - bytes) return KVR_ERR_INVALID_ARG;
  return launch_stand_in(compute, offset, bytes, static_cast<cudaStream_t>(stream));
}

static int check_layer(const kvr_dims *dims, const kvr_layer &L, int32_t top_k, float tau) {
  int rc = check_spec(dims, L.st, L.q, L.summ, L.corrected, L.cbar_opt, L.sel_used, tau);
  if (rc) return rc;
  if (!L.out || !L.sel_used_idx) return KVR_ERR_INVALID_ARG;
  if (!aligned16(L.out) || !aligned16(L.sel_used_idx)) return KVR_ERR_ALIGN;
  if (L.host) {
    if ((rc = check_wset(dims, L.wset, top_k))) return rc;
    if (!L.host->k_host || !L.host->v_host || !L.ev[0] || !L.ev[1] || !L.ev[2])
      return KVR_ERR_INVALID_ARG;
    if (!aligned16(L.host->k_host) || !aligned16(L.host->v_host)) return KVR_ERR_ALIGN;
  } else {
    if (!L.page_table || !L.k_pool || !L.v_pool) return KVR_ERR_INVALID_ARG;
    if (!aligned16(L.page_table) || !aligned16(L.k_pool) || !aligned16(L.v_pool))
      return KVR_ERR_ALIGN;
  }
  return check_ws(L.ws, L.ws_bytes, select_ws_bytes(dims) + attn_ws_bytes(dims, top_k));
}

int kvr_pipeline_step(const kvr_dims *dims, int32_t n_layers, kvr_layer *layers,
                      const kvr_stand_in *compute, int32_t top_k, float tau, float scale,
                      void *stream, void *side_stream, void *prefetch_stream,
                      void *const *marks) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_topk(dims, top_k))) return rc;
  if (n_layers <= 0 || !layers || std::isnan(scale)) return KVR_ERR_INVALID_ARG;
  if (compute && (rc = check_stand_in(compute))) return rc;
  for (int l = 0; l < n_layers; ++l)
    if ((rc = check_layer(dims, layers[l], top_k, tau))) return rc;
  if (marks)
    for (int64_t i = 0; i < static_cast<int64_t>(n_layers) * KVR_PIPE_MARKS; ++i)
      if (!marks[i]) return KVR_ERR_INVALID_ARG;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t side = static_cast<cudaStream_t>(side_stream);
  cudaStream_t pf = static_cast<cudaStream_t>(prefetch_stream);
  auto record = [](void *ev, cudaStream_t st) {
    const cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(ev), st);
    return e == cudaSuccess ? KVR_OK : cuda_fail(e, "pipeline event record");
  };
  auto wait = [](cudaStream_t st, void *ev) {
    const cudaError_t e = cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(ev), 0);
    return e == cudaSuccess ? KVR_OK : cuda_fail(e, "pipeline stream wait");
  };
  // timing marks: while the stream is being captured they are recorded as
  // external events, so that the graph records them on every replay (the
  // flag is refused outside a capture)
  auto mark = [&](int l, int m, cudaStream_t st) {
    if (!marks) return KVR_OK;
    cudaEvent_t ev = static_cast<cudaEvent_t>(marks[static_cast<int64_t>(l) * KVR_PIPE_MARKS + m]);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e == cudaSuccess)
      e = cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal)
                                              : cudaEventRecord(ev, st);
    return e == cudaSuccess ? KVR_OK : cuda_fail(e, "pipeline timing mark");
  };
  const uint64_t qkv = compute ? compute->qkv_bytes : 0;
  const uint64_t post = compute ? compute->post_bytes : 0;
#define KVR_TRY(x) \
  if ((rc = (x))) return rc
  for (int l = 0; l < n_layers; ++l) {
    kvr_layer &L = layers[l];
    const AttnWs aw = carve_attn(dims, top_k, static_cast<uint8_t *>(L.ws) + select_ws_bytes(dims));
    KVR_TRY(mark(l, 0, s));
    KVR_TRY(launch_stand_in(compute, 0, qkv, s));
    KVR_TRY(mark(l, 1, s));
    if (!L.host) {
      // kvr_speculative_step: the selection, whose speculative prologue
      // announces the reused heads' page ids, then the attention, whose
      // reused units start before the selection ends.  One chain of
      // dependent launches on `stream`; a mark between its kernels would
      // cut it, so this layer's side marks come first and marks 2-4 after
      // the attention.
      KVR_TRY(mark(l, 7, s));
      KVR_TRY(mark(l, 8, s));
      KVR_TRY(mark(l, 9, s));
      KVR_TRY(mark(l, 10, s));
      const unsigned long long tag = next_ready_tag();
      KVR_TRY(spec_select_impl(dims, L.st, L.q, L.summ, L.page_table, top_k, tau, L.corrected,
                               L.cbar_opt, L.sel_used, L.sel_used_idx, nullptr, 0, L.ws, s, true,
                               aw.ready, tag));
      L.st->step += 1;
      AttnLen early;
      early.ready = aw.ready;
      early.ready_tag = tag;
      KVR_TRY(launch_attn(dims, L.q, L.k_pool, L.v_pool, dims->n_phys_pages, L.sel_used_idx, top_k,
                          scale, nullptr, 0, aw, L.out, s, true, early));
      KVR_TRY(mark(l, 2, s));
      KVR_TRY(mark(l, 3, s));
      KVR_TRY(mark(l, 4, s));
    } else {
      // this layer's maps and slots as the previous step's prefetch left them
      KVR_TRY(wait(s, L.ev[2]));
      KVR_TRY(spec_select_impl(dims, L.st, L.q, L.summ, nullptr, top_k, tau, L.corrected,
                               L.cbar_opt, L.sel_used, L.sel_used_idx, L.wset->page2slot,
                               L.wset->n_slots, L.ws, s, false));
      L.st->step += 1;
      KVR_TRY(mark(l, 2, s));
      KVR_TRY(record(L.ev[0], s));
      // side stream: the pages the corrected heads need now
      KVR_TRY(wait(side, L.ev[0]));
      KVR_TRY(mark(l, 7, side));
      KVR_TRY(launch_recall(dims, L.host, L.wset, L.st->sel_prev, L.sel_used, L.corrected, top_k,
                            L.sel_used_idx, L.n_copied_opt, side, 2));
      KVR_TRY(mark(l, 8, side));
      KVR_TRY(record(L.ev[1], side));
      // prefetch stream, after it: the other heads' new selection (next step)
      KVR_TRY(wait(pf, L.ev[1]));
      KVR_TRY(mark(l, 9, pf));
      KVR_TRY(launch_recall(dims, L.host, L.wset, L.st->sel_prev, L.sel_used, L.corrected, top_k,
                            L.sel_used_idx, L.n_copied_opt, pf, 1));
      KVR_TRY(mark(l, 10, pf));
      KVR_TRY(record(L.ev[2], pf));
      const int64_t n_phys = static_cast<int64_t>(dims->batch) * L.wset->n_slots;
      KVR_TRY(launch_attn(dims, L.q, L.wset->k_slots, L.wset->v_slots, n_phys, L.sel_used_idx,
                          top_k, scale, L.corrected, 1, aw, L.out, s, false));
      KVR_TRY(mark(l, 3, s));
      KVR_TRY(wait(s, L.ev[1]));
      KVR_TRY(mark(l, 4, s));
      KVR_TRY(launch_attn(dims, L.q, L.wset->k_slots, L.wset->v_slots, n_phys, L.sel_used_idx,
                          top_k, scale, L.corrected, 2, aw, L.out, s, false));
    }
    KVR_TRY(mark(l, 5, s));
    KVR_TRY(launch_stand_in(compute, qkv, post, s));
    KVR_TRY(mark(l, 6, s));
  }
#undef KVR_TRY
  return KVR_OK;
}

int kvr_get_status(void *stream, uint32_t *status_out) {
  if (!status_out) return KVR_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "status sync");
  uint32_t v = 0;
  e = cudaMemcpyFromSymbolAsync(&v, g_status, sizeof v, 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  const uint32_t zero = 0;
  e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "status clear");
  *status_out = v;
  return KVR_OK;
}

int kvr_set_wait_limit(uint64_t ns) {
  g_wait_limit.store(ns ? ns : kWaitNs, std::memory_order_relaxed);
  return KVR_OK;
}

int kvr_stream_wait(void *stream, uint64_t timeout_us) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    const cudaError_t e = cudaStreamQuery(s);
    if (e == cudaSuccess) return KVR_OK;
    if (e != cudaErrorNotReady) return cuda_fail(e, "stream wait");
    // "not ready" is a state, not an error: keep it out of the launch checks
    if (cudaPeekAtLastError() == cudaErrorNotReady) (void)cudaGetLastError();
    const auto us = std::chrono::duration_cast<std::chrono::microseconds>(
                        std::chrono::steady_clock::now() - t0)
                        .count();
    if (static_cast<uint64_t>(us) >= timeout_us) return KVR_ERR_TIMEOUT;
    std::this_thread::yield();
  }
}

const char *kvr_error_string(int code) {
  switch (code) {
    case KVR_OK: return "ok";
    case KVR_ERR_INVALID_ARG: return "invalid argument (null pointer, bad size or enum)";
    case KVR_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case KVR_ERR_ALIGN: return "pointer not 16-byte aligned";
    case KVR_ERR_WORKSPACE: return "workspace missing or too small";
    case KVR_ERR_CUDA: return g_err_text[0] ? g_err_text : "CUDA error";
    case KVR_ERR_TIMEOUT: return "host-side wait timed out";
    case KVR_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than the fixed array of the allocation-free entry point";
    default: return "unknown error code";
  }
}

uint64_t kvr_kv_bytes(int64_t n_layers, int64_t n_kv_heads, int64_t head_dim, int64_t n_tokens,
                      int64_t bytes_per_elem) {
  if (n_layers < 0 || n_kv_heads < 0 || head_dim < 0 || n_tokens < 0 || bytes_per_elem < 0) return 0;
  unsigned __int128 v = 2;
  for (int64_t f : {n_layers, n_kv_heads, head_dim, n_tokens, bytes_per_elem}) {
    v *= static_cast<unsigned __int128>(f);
    if (v > static_cast<unsigned __int128>(UINT64_MAX)) return 0;
  }
  return static_cast<uint64_t>(v);
}

}  // extern "C"

// ---------------------------------------------------------------- allocation-free selection
//
// kvr_select_pages_noalloc: the selection kernels with their scratch (the
// score rows) in this fixed device array instead of a caller
// workspace, for callers that may not allocate device memory.  Host code
// must not pass the array's name to a kernel (on the host it only stands in
// for the symbol); the device address is looked up on every call below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KVR_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the scratch array on the current device.  Looked up on
// every call (a host-side query that allocates nothing), so an address from
// a context that was since destroyed (cudaDeviceReset) is never reused.
int noalloc_scratch(void **out) {
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "scratch symbol address");
  *out = p;
  return KVR_OK;
}

}  // namespace

extern "C" int kvr_select_pages_noalloc(const kvr_dims *dims, const uint16_t *q,
                                        const uint16_t *summ, const int32_t *page_table,
                                        int32_t top_k, int32_t *sel, int32_t *sel_phys,
                                        float *scores_opt, void *stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_topk(dims, top_k))) return rc;
  if (!q || !summ || !page_table || !sel) return KVR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(summ) || !aligned16(page_table) || !aligned16(sel) ||
      (sel_phys && !aligned16(sel_phys)) || (scores_opt && !aligned16(scores_opt)))
    return KVR_ERR_ALIGN;
  const size_t need = select_ws_bytes(dims);
  if (need > KVR_NOALLOC_SCRATCH_BYTES) return KVR_ERR_SCRATCH_LIMIT;
  void *scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const SelectWs w = carve_select(dims, static_cast<uint8_t *>(scratch));
  return launch_select(dims, q, summ, page_table, top_k, w, sel, sel_phys, scores_opt, no_spec(),
                       st);
}
