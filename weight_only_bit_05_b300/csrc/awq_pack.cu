// Scaled group round-to-nearest with zero point, and packing.
//
// "AWQ量化实战：无需重训，把大模型压进4bit显存" §1.1 (round to nearest), §2.1 (the
// channel is the input dimension of the out x in weight), §2.3 (128
// consecutive input channels share one step); "大模型量化部署实战：GPTQ与AWQ算法",
// section 大模型量化的核心原理与位宽选择 (a scale plus a zero point per group).
//
// One warp owns row n and 8 consecutive groups (1024 input channels, the span
// of one zero-point word).  Lane l holds 32 consecutive weights (a quarter
// group): four lanes reduce a group's min/max with two shuffles, every lane
// decides its 32 codes in fp32 with IEEE division and round-half-even (the
// same operations, in the same precision, as the definition), writes one
// 16-byte word quad, and the warp ORs the 8 zero points into one word.
#include "awq_internal.h"

namespace awq {
namespace {

__global__ void __launch_bounds__(256)
    quant_pack_kernel(const __half* __restrict__ W, const float* __restrict__ s_c, int N, int K,
                      uint32_t* __restrict__ qweight, __half* __restrict__ scales,
                      uint32_t* __restrict__ zeros) {
  const int G = K / kGroup;
  const int units = (G + 7) / 8;                  // zero-point words per row
  const int gw = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (gw >= N * units) return;
  const int lane = threadIdx.x & 31;
  const int n = gw / units, u = gw - n * units;
  const int k0 = u * 1024 + lane * 32;            // this lane's first input channel
  const bool valid = k0 < K;                      // whole quarter groups only (K % 128 == 0)

  float w[32];
  if (valid) {
    const uint4* src = reinterpret_cast<const uint4*>(W + static_cast<size_t>(n) * K + k0);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 raw = __ldg(src + v);
      const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(h[j]);
        w[v * 8 + 2 * j] = f.x;
        w[v * 8 + 2 * j + 1] = f.y;
      }
    }
    if (s_c) {
      const float4* sc = reinterpret_cast<const float4*>(s_c + k0);
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const float4 s = __ldg(sc + v);
        w[4 * v + 0] = __fmul_rn(w[4 * v + 0], s.x);
        w[4 * v + 1] = __fmul_rn(w[4 * v + 1], s.y);
        w[4 * v + 2] = __fmul_rn(w[4 * v + 2], s.z);
        w[4 * v + 3] = __fmul_rn(w[4 * v + 3], s.w);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = 0.f;
  }

  float mn = w[0], mx = w[0];
#pragma unroll
  for (int i = 1; i < 32; ++i) {
    mn = fminf(mn, w[i]);
    mx = fmaxf(mx, w[i]);
  }
  // min/max over the 4 lanes of the group (lanes 4g..4g+3)
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }

  float s32 = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
  s32 = fminf(fmaxf(s32, 6.103515625e-05f), 65504.0f);   // [2^-14, 65504]
  const __half s16 = __float2half_rn(s32);
  const float s = __half2float(s16);
  const float z = fminf(fmaxf(rintf(__fdiv_rn(-mn, s)), 0.f), 15.f);

  uint32_t words[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float q = fminf(fmaxf(rintf(__fdiv_rn(w[v * 8 + i], s)) + z, 0.f), 15.f);
      word |= static_cast<uint32_t>(q) << (4 * i);
    }
    words[v] = word;
  }

  const int g = k0 / kGroup;
  if (valid) {
    uint4* dst = reinterpret_cast<uint4*>(qweight + static_cast<size_t>(n) * (K / 8) + k0 / 8);
    *dst = make_uint4(words[0], words[1], words[2], words[3]);
    if ((lane & 3) == 0) scales[static_cast<size_t>(n) * G + g] = s16;
  }
  const uint32_t zc = (valid && (lane & 3) == 0) ? static_cast<uint32_t>(z) << (4 * (g & 7)) : 0u;
  const uint32_t zword = __reduce_or_sync(0xffffffffu, zc);
  if (lane == 0) zeros[static_cast<size_t>(n) * units + u] = zword;
}

}  // namespace

int launch_pack(const __half* W, const float* s_c, int N, int K, uint32_t* qweight,
                __half* scales, uint32_t* zeros, cudaStream_t st) {
  const int units = (K / kGroup + 7) / 8;
  const int64_t warps = static_cast<int64_t>(N) * units;
  const int64_t blocks = (warps + 7) / 8;
  quant_pack_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(W, s_c, N, K, qweight, scales,
                                                                   zeros);
  AWQ_CUDA_TRY_LAUNCH("quant_pack_kernel");
  return AWQ_OK;
}

}  // namespace awq
