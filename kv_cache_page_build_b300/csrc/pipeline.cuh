// pipeline.cuh -- the stand-in for the rest of a transformer layer in the
// multi-layer decode pipeline (kvr_pipeline_step).
//
// Source: FreeKV (technical summary), section 2.1: speculative retrieval
// overlaps the selection and recall of a layer with that layer's attention
// and FFN and with the next layer's QKV projection.  Those projections are
// not part of this library; at decode batch sizes a projection is bound by
// reading its weights once, so the pipeline models each one by a kernel that
// streams the same number of bytes from HBM.
//
// k_stand_in reads n16 16-byte words (grid-stride, four loads in flight per
// thread, not allocated in L1) and adds their 32-bit lanes, modulo 2^32, into
// *sink: the sum keeps the loads live and is independent of the order in
// which the CTAs finish, so a caller can check it exactly.
#pragma once

#include "common.cuh"

namespace kvr {

constexpr int kStandInThreads = 512;
constexpr int kStandInCPS = 2;  // CTAs per SM

__global__ void __launch_bounds__(kStandInThreads)
    k_stand_in(const uint4 *__restrict__ w, uint64_t n16, uint32_t *__restrict__ sink) {
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kStandInThreads;
  uint64_t i = static_cast<uint64_t>(blockIdx.x) * kStandInThreads + threadIdx.x;
  uint32_t acc = 0;
  constexpr int U = 4;
  for (; i + (U - 1) * stride < n16; i += U * stride) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = ld_stream_v4(w + i + u * stride);
#pragma unroll
    for (int u = 0; u < U; ++u) acc += v[u].x + v[u].y + v[u].z + v[u].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = ld_stream_v4(w + i);
    acc += v.x + v.y + v.z + v.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0 && acc != 0) atomicAdd(sink, acc);
}

}  // namespace kvr
