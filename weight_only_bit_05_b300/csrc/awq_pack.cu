// Scaled group round-to-nearest, and packing.
//
// "AWQ量化实战：无需重训，把大模型压进4bit显存" §1.1 (round to nearest), §2.1 (the
// channel is the input dimension of the out x in weight), §2.3 (GS = 128,
// also 64 or 32, consecutive input channels share one step), §3.3 (zero
// point off is the symmetric form; 8 bits is the conservative width);
// "大模型量化部署实战：GPTQ与AWQ算法", section 大模型量化的核心原理与位宽选择 (a scale
// plus a zero point per group; int4 spans -8..7).
//
// One warp owns row n and 1024 consecutive input channels.  Lane l holds 32
// consecutive weights: GS/32 lanes reduce a group's min/max with shuffles,
// every lane decides its 32 codes in fp32 with IEEE division and
// round-half-even (the same operations, in the same precision, as the
// definition), writes its 32 codes as one or two 16-byte stores, and the
// warp ORs the groups' zero points into their words.
#include "awq_internal.h"

namespace awq {
namespace {

// Shrink ratio i of an n-point clipping grid: fp32(1 - 0.5 i / n), the fp64
// operations in the order of the definition.
__device__ __forceinline__ float clip_ratio(int i, int n) {
  return __double2float_rn(__dsub_rn(1.0, __ddiv_rn(__dmul_rn(0.5, static_cast<double>(i)),
                                                    static_cast<double>(n))));
}

// clip_idx (optional, uint8 [N][G]): the group's range is shrunk by
// clip_ratio(clip_idx[n][g], n_clip) before its step and zero point are set;
// the codes then clamp, which clips the weights outside the shrunk range.
template <int BITS, int GS, bool ZP>
__global__ void __launch_bounds__(256)
    quant_pack_kernel(const __half* __restrict__ W, const float* __restrict__ s_c, int N, int K,
                      uint32_t* __restrict__ qweight, __half* __restrict__ scales,
                      uint32_t* __restrict__ zeros, const uint8_t* __restrict__ clip_idx,
                      int n_clip) {
  constexpr int kPerWord = 32 / BITS;             // codes per packed word
  constexpr int kQmax = (1 << BITS) - 1;
  constexpr int kHalf = 1 << (BITS - 1);
  constexpr int kLanesPerGroup = GS / 32;
  constexpr int kZWords = (1024 / GS) / kPerWord;   // zero-point words per warp span
  const int G = K / GS;
  const int ZW = (G + kPerWord - 1) / kPerWord;   // zero-point words per row
  const int units = (K + 1023) / 1024;            // warp spans per row
  const int gw = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (gw >= N * units) return;
  const int lane = threadIdx.x & 31;
  const int n = gw / units, u = gw - n * units;
  const int k0 = u * 1024 + lane * 32;            // this lane's first input channel
  const bool valid = k0 < K;                      // whole lanes only (K % 128 == 0)

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
  // min/max over the lanes of the group
#pragma unroll
  for (int off = 1; off < kLanesPerGroup; off <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }

  float amax = fmaxf(fabsf(mn), fabsf(mx));
  if (clip_idx && valid) {
    const float r = clip_ratio(clip_idx[static_cast<size_t>(n) * G + k0 / GS], n_clip);
    mn = __fmul_rn(mn, r);
    mx = __fmul_rn(mx, r);
    amax = __fmul_rn(amax, r);
  }
  float s32 = ZP ? __fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(kQmax))
                 : __fdiv_rn(amax, static_cast<float>(kHalf - 1));
  s32 = fminf(fmaxf(s32, 6.103515625e-05f), 65504.0f);   // [2^-14, 65504]
  const __half s16 = __float2half_rn(s32);
  const float s = __half2float(s16);
  const float z = ZP ? fminf(fmaxf(rintf(__fdiv_rn(-mn, s)), 0.f), static_cast<float>(kQmax))
                     : static_cast<float>(kHalf);

  constexpr int kWords = 32 / kPerWord;           // packed words of this lane
  uint32_t words[kWords];
#pragma unroll
  for (int v = 0; v < kWords; ++v) {
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < kPerWord; ++i) {
      const float r = rintf(__fdiv_rn(w[v * kPerWord + i], s));
      const float q = ZP ? fminf(fmaxf(r + z, 0.f), static_cast<float>(kQmax))
                         : fminf(fmaxf(r, static_cast<float>(-kHalf)),
                                 static_cast<float>(kHalf - 1)) + static_cast<float>(kHalf);
      word |= static_cast<uint32_t>(q) << (BITS * i);
    }
    words[v] = word;
  }

  const int g = k0 / GS;
  const bool leader = valid && (lane % kLanesPerGroup) == 0;
  if (valid) {
    uint4* dst = reinterpret_cast<uint4*>(qweight + static_cast<size_t>(n) * (K / kPerWord) +
                                          k0 / kPerWord);
#pragma unroll
    for (int v = 0; v < kWords / 4; ++v)
      dst[v] = make_uint4(words[4 * v], words[4 * v + 1], words[4 * v + 2], words[4 * v + 3]);
    if (leader) scales[static_cast<size_t>(n) * G + g] = s16;
  }
  // the zero points of this warp's groups, kPerWord to a word
  const int gl = g - u * (1024 / GS);             // group index within the warp span
#pragma unroll
  for (int zw = 0; zw < kZWords; ++zw) {
    const uint32_t zc = (leader && gl / kPerWord == zw)
                            ? static_cast<uint32_t>(z) << (BITS * (gl % kPerWord)) : 0u;
    const uint32_t zword = __reduce_or_sync(0xffffffffu, zc);
    const int col = u * kZWords + zw;
    if (lane == 0 && col < ZW) zeros[static_cast<size_t>(n) * ZW + col] = zword;
  }
}

}  // namespace

int launch_pack(const __half* W, const float* s_c, int N, int K, uint32_t* qweight,
                __half* scales, uint32_t* zeros, cudaStream_t st, int w_bit, int group,
                bool zero_point, const uint8_t* clip_idx, int n_clip) {
  const int units = (K + 1023) / 1024;
  const int64_t warps = static_cast<int64_t>(N) * units;
  const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
#define AWQ_PACK_CASE(B, GS, ZP)                                                         \
  if (w_bit == B && group == GS && zero_point == ZP) {                                   \
    quant_pack_kernel<B, GS, ZP><<<blocks, 256, 0, st>>>(W, s_c, N, K, qweight, scales, \
                                                         zeros, clip_idx, n_clip);      \
    AWQ_CUDA_TRY_LAUNCH("quant_pack_kernel");                                            \
    return AWQ_OK;                                                                       \
  }
  AWQ_PACK_CASE(4, 128, true)
  AWQ_PACK_CASE(4, 64, true)
  AWQ_PACK_CASE(4, 32, true)
  AWQ_PACK_CASE(4, 128, false)
  AWQ_PACK_CASE(4, 64, false)
  AWQ_PACK_CASE(4, 32, false)
  AWQ_PACK_CASE(8, 128, true)
  AWQ_PACK_CASE(8, 64, true)
  AWQ_PACK_CASE(8, 32, true)
  AWQ_PACK_CASE(8, 128, false)
  AWQ_PACK_CASE(8, 64, false)
  AWQ_PACK_CASE(8, 32, false)
#undef AWQ_PACK_CASE
  set_error("awq_pack: w_bit = %d, group = %d, zero_point = %d is not supported", w_bit, group,
            static_cast<int>(zero_point));
  return AWQ_ERR_UNSUPPORTED;
}

namespace {
__global__ void stream_fence_kernel() {}
}  // namespace

// An empty kernel launched without programmatic dependent launch: it starts
// only once the kernels before it on the stream have completed and their
// writes are visible, so a following kernel that reads weights before its
// dependency wait (the decode matmul) overlaps this kernel, never the pack.
int launch_stream_fence(cudaStream_t st) {
  stream_fence_kernel<<<1, 32, 0, st>>>();
  AWQ_CUDA_TRY_LAUNCH("stream_fence_kernel");
  return AWQ_OK;
}

}  // namespace awq
