// Measurement aid (not a step of the method): a plain streaming read of a
// buffer, launched like the decode matmul (programmatic dependent launch), so
// that a chain of such launches over the same weight bytes gives the ceiling
// that HBM and launch-to-launch overlap allow a chain of decode matmuls.
#include "awq_internal.h"

namespace awq {
namespace {

// Reads [p, p + n16 * 16) with 16-byte streaming loads, eight in flight per
// thread, and folds them into one word per CTA (written only when it hits a
// value no buffer of real weights produces, so the loads cannot be dropped).
// read_first: the reads are issued before griddepcontrol.wait (weights do
// not depend on the previous kernel), else after it.
__global__ void __launch_bounds__(512, 1)
    stream_read_kernel(const uint4* __restrict__ p, size_t n16, int read_first,
                       unsigned* __restrict__ out) {
  if (!read_first) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  uint32_t acc = 0;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 7 * stride < n16; i += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldcs(p + i + u * stride);
#pragma unroll
    for (int u = 0; u < 8; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = __ldcs(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (read_first) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (acc == 0x9E3779B9u) out[blockIdx.x] = acc;
}

}  // namespace

int launch_stream_read(const void* buf, size_t bytes, int read_first, unsigned* out,
                       cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sm_count(), 1, 1);
  cfg.blockDim = dim3(512, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  AWQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, stream_read_kernel, static_cast<const uint4*>(buf),
                                  bytes / 16, read_first, out));
  return AWQ_OK;
}

}  // namespace awq
