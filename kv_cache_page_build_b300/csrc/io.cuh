// io.cuh -- host-buffer input of a decode step (kvr_speculative_step_host).
//
// Source: FreeKV (technical summary), section 2.2: the system keeps the
// decode step's data movement off the critical path.  A step's query comes
// from page-locked host memory and its output goes back there; each is a few
// tens of KiB, so a copy-engine transfer costs far more in the hand-offs
// between the copy engine and the kernels around it than in moving the bytes.
// Instead the step's first kernel reads the query through the host mapping
// and stages it in device memory, and the attention stores its output
// through the host mapping.
//
// k_stage_in copies n16 16-byte words from page-locked host memory into
// device memory.  Launched as a programmatic dependent launch, it issues its
// first host reads before the dependency wait, so that their latency
// overlaps the kernel before it (the host buffer is no kernel's output, and
// the staged copy may still be read by the previous step until the wait);
// it stores only after the wait.  It does not let the next kernel launch
// early: that kernel reads the staged query through the read-only path,
// which is only safe for data no kernel still running writes.
#pragma once

#include "common.cuh"

namespace kvr {

constexpr int kStageThreads = 256;

__global__ void __launch_bounds__(kStageThreads)
    k_stage_in(const uint4 *__restrict__ host, uint4 *__restrict__ dst, uint64_t n16) {
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kStageThreads;
  uint64_t i = static_cast<uint64_t>(blockIdx.x) * kStageThreads + threadIdx.x;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (i < n16) v = host[i];  // through the host mapping, before the wait
  pdl_wait();
  if (i < n16) dst[i] = v;
  for (i += stride; i < n16; i += stride) dst[i] = host[i];
}

}  // namespace kvr
