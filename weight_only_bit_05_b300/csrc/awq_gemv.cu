// W4A16 GEMV for M <= 8 tokens on CUDA cores.
//
// "awq-quantization（AWQ量化技术）Skill" page, section 主要功能和特点: a GEMV kernel
// serves batch-1 token generation; "AWQ量化实战" §3.4: decoding is bound by the
// bandwidth of reading the weights.  So this kernel is organised around
// streaming the packed codes from HBM exactly once:
//
//  * one warp owns two output rows; lane l reads 16 bytes (4 packed words = 32
//    codes = a quarter of a group) of each row per iteration, so a warp reads
//    512 contiguous bytes of a row per load instruction;
//  * the scaled activations x~ = fp32(x) * inv_s of the CTA's K slice are
//    computed once per CTA into shared memory, laid out so that the 32 lanes
//    read 32 consecutive 16-byte vectors (no bank conflicts) and reused by
//    every row of the CTA;
//  * codes become exact fp32 numbers 2^23 + q by a byte permute into the
//    exponent of 2^23; subtracting 2^23 + z gives q - z exactly, and the
//    products x~ (q - z) are summed in fp32 with packed two-wide FMAs; the
//    group step s multiplies each lane's quarter-group sum;
//  * lanes are reduced with warp shuffles; when K is split across CTAs (to
//    occupy every SM, or to keep the x~ slice small) the CTAs of one row tile
//    form a thread-block cluster and the partial sums are added in rank order
//    through distributed shared memory (deterministic, no global scratch).
#include <cooperative_groups.h>

#include "awq_internal.h"

namespace cg = cooperative_groups;

namespace awq {
namespace {

constexpr int kWarps = 8;
constexpr int kRowsPerWarp = 2;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;
constexpr int kMaxSplit = 8;
constexpr int kSmemFast = 48 * 1024;
constexpr int kSmemMax = 200 * 1024;

__device__ __forceinline__ float magic_code(uint32_t v, uint32_t sel) {
  // byte `sel & 3` of v into the low mantissa byte of 2^23: the value 2^23 + byte
  return __uint_as_float(__byte_perm(v, 0x4B000000u, sel));
}

// Adds x~[k0..k7] * (q[k0..k7] - z) to acc (two fp32 lanes) for one packed word.
template <int MM>
__device__ __forceinline__ void word_dot(uint32_t w, float2 nzb, const float4 (&x)[MM][2],
                                         float2 (&acc)[MM]) {
  const uint32_t lo = w & 0x0F0F0F0Fu;          // codes of k0, k2, k4, k6
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;   // codes of k1, k3, k5, k7
  const float2 q01 = __fadd2_rn(make_float2(magic_code(lo, 0x7440), magic_code(hi, 0x7440)), nzb);
  const float2 q23 = __fadd2_rn(make_float2(magic_code(lo, 0x7441), magic_code(hi, 0x7441)), nzb);
  const float2 q45 = __fadd2_rn(make_float2(magic_code(lo, 0x7442), magic_code(hi, 0x7442)), nzb);
  const float2 q67 = __fadd2_rn(make_float2(magic_code(lo, 0x7443), magic_code(hi, 0x7443)), nzb);
#pragma unroll
  for (int m = 0; m < MM; ++m) {
    acc[m] = __ffma2_rn(make_float2(x[m][0].x, x[m][0].y), q01, acc[m]);
    acc[m] = __ffma2_rn(make_float2(x[m][0].z, x[m][0].w), q23, acc[m]);
    acc[m] = __ffma2_rn(make_float2(x[m][1].x, x[m][1].y), q45, acc[m]);
    acc[m] = __ffma2_rn(make_float2(x[m][1].z, x[m][1].w), q67, acc[m]);
  }
}

// Shared-memory slot (in float4) of the 4 activations starting at local k.
__device__ __forceinline__ int xs_slot(int kl) {
  const int t = kl >> 10, lane = (kl >> 5) & 31, v = (kl >> 2) & 7;
  return (t * 8 + v) * 32 + lane;
}

template <int MM>
__global__ void __launch_bounds__(kWarps * 32)
    gemv_kernel(const __half* __restrict__ X, const uint32_t* __restrict__ qweight,
                const __half* __restrict__ scales, const uint32_t* __restrict__ zeros,
                const float* __restrict__ inv_s, int N, int K, int KS, int xs_stride,
                __half* __restrict__ Y) {
  extern __shared__ float4 xs[];   // [MM][xs_stride] float4, permuted
  __shared__ float red[MM][kRowsPerCta];

  const int split = blockIdx.y;
  const int kbeg = split * KS;
  const int klen = min(K - kbeg, KS);   // multiple of 128

  // x~ = fp32(x) * inv_s for this slice, rounded to fp32 once
  const int q4 = klen >> 2;
  for (int v = threadIdx.x; v < MM * q4; v += blockDim.x) {
    const int m = v / q4, kl = (v - m * q4) << 2;
    const uint2 xr = __ldg(reinterpret_cast<const uint2*>(X + static_cast<size_t>(m) * K + kbeg + kl));
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&xr.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&xr.y));
    float4 o = make_float4(a.x, a.y, b.x, b.y);
    if (inv_s) {
      const float4 is = __ldg(reinterpret_cast<const float4*>(inv_s + kbeg + kl));
      o.x = __fmul_rn(o.x, is.x);
      o.y = __fmul_rn(o.y, is.y);
      o.z = __fmul_rn(o.z, is.z);
      o.w = __fmul_rn(o.w, is.w);
    }
    xs[m * xs_stride + xs_slot(kl)] = o;
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = K / kGroup, ZW = (G + 7) / 8, KW = K / 8;
  const int row0 = blockIdx.x * kRowsPerCta + warp * kRowsPerWarp;
  float acc[kRowsPerWarp][MM];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
    for (int m = 0; m < MM; ++m) acc[r][m] = 0.f;

  // iterations in which this lane has a quarter group inside the slice
  const int nit = (klen - lane * 32 + 1023) >> 10;
  for (int t = 0; t < nit; t += 2) {
    uint4 wq[2][kRowsPerWarp];
    float s[2][kRowsPerWarp];
    float2 nzb[2][kRowsPerWarp];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int kl = ((t + u) << 10) + (lane << 5);
      const int k = kbeg + kl, g = k >> 7;
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        const int row = row0 + r;
        if (t + u < nit && row < N) {
          wq[u][r] = __ldcs(reinterpret_cast<const uint4*>(qweight + static_cast<size_t>(row) * KW + (k >> 3)));
          s[u][r] = __half2float(scales[static_cast<size_t>(row) * G + g]);
          const uint32_t zw = __ldg(zeros + static_cast<size_t>(row) * ZW + (g >> 3));
          const float zb = -(8388608.0f + static_cast<float>((zw >> ((g & 7) * 4)) & 15u));
          nzb[u][r] = make_float2(zb, zb);
        } else {
          wq[u][r] = make_uint4(0, 0, 0, 0);
          s[u][r] = 0.f;
          nzb[u][r] = make_float2(-8388608.0f, -8388608.0f);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (t + u >= nit) break;
      const int kl = ((t + u) << 10) + (lane << 5);
      float2 part[kRowsPerWarp][MM];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int m = 0; m < MM; ++m) part[r][m] = make_float2(0.f, 0.f);
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {
        float4 xv[MM][2];
#pragma unroll
        for (int m = 0; m < MM; ++m) {
          xv[m][0] = xs[m * xs_stride + xs_slot(kl + wd * 8)];
          xv[m][1] = xs[m * xs_stride + xs_slot(kl + wd * 8 + 4)];
        }
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
          const uint32_t w = wd == 0 ? wq[u][r].x : wd == 1 ? wq[u][r].y : wd == 2 ? wq[u][r].z : wq[u][r].w;
          word_dot<MM>(w, nzb[u][r], xv, part[r]);
        }
      }
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int m = 0; m < MM; ++m) acc[r][m] = fmaf(s[u][r], part[r][m].x + part[r][m].y, acc[r][m]);
    }
  }

#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
    for (int m = 0; m < MM; ++m) {
      float v = acc[r][m];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      acc[r][m] = v;
    }

  if (gridDim.y == 1) {
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r)
        if (row0 + r < N)
#pragma unroll
          for (int m = 0; m < MM; ++m)
            Y[static_cast<size_t>(m) * N + row0 + r] = __float2half_rn(acc[r][m]);
    }
    return;
  }

  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
      for (int m = 0; m < MM; ++m) red[m][warp * kRowsPerWarp + r] = acc[r][m];
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  if (cluster.block_rank() == 0) {
    const int nsplit = gridDim.y;
    for (int i = threadIdx.x; i < MM * kRowsPerCta; i += blockDim.x) {
      float sum = 0.f;
      for (int rk = 0; rk < nsplit; ++rk) sum += cluster.map_shared_rank(&red[0][0], rk)[i];
      const int m = i / kRowsPerCta, row = blockIdx.x * kRowsPerCta + (i - m * kRowsPerCta);
      if (row < N) Y[static_cast<size_t>(m) * N + row] = __float2half_rn(sum);
    }
  }
  cluster.sync();   // keep every CTA's shared memory alive until rank 0 has read it
}

int num_sms() {
  static int cached = -1;
  if (cached < 0) {
    int dev = 0, n = 148;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      cached = n;
    else
      cached = 148;
  }
  return cached;
}

template <int MM>
int launch_mm(const __half* X, const uint32_t* qweight, const __half* scales,
              const uint32_t* zeros, const float* inv_s, int N, int K, __half* Y,
              cudaStream_t st) {
  const int ntile = (N + kRowsPerCta - 1) / kRowsPerCta;
  auto round_up = [](int v, int m) { return (v + m - 1) / m * m; };
  // slice length: keep the x~ slice at <= 48 KB when possible (occupancy)
  // (x~ takes MM * 4 bytes per input channel; slices are multiples of 1024)
  auto cap_for = [](int bytes) { return max(1024, (bytes / (MM * 4)) / 1024 * 1024); };
  int ks_cap = cap_for(kSmemFast);
  int nsplit = (K + ks_cap - 1) / ks_cap;
  if (nsplit > kMaxSplit) {
    ks_cap = cap_for(kSmemMax);
    nsplit = (K + ks_cap - 1) / ks_cap;
    if (nsplit > kMaxSplit) {
      set_error("awq_gemv: K = %d is too large for M = %d (use awq_gemm)", K, MM);
      return AWQ_ERR_SHAPE;
    }
  }
  // split further to give every SM at least two CTAs
  const int target = (2 * num_sms() + ntile - 1) / ntile;
  const int by_k = K / 1024 > 0 ? K / 1024 : 1;
  nsplit = max(nsplit, min(min(target, kMaxSplit), by_k));
  const int KS = round_up((K + nsplit - 1) / nsplit, kGroup);
  nsplit = (K + KS - 1) / KS;
  const int xs_stride = round_up(KS, 1024) / 4;
  const size_t smem = static_cast<size_t>(MM) * xs_stride * sizeof(float4);

  static bool attr_set = false;
  if (!attr_set) {
    AWQ_CUDA_TRY(cudaFuncSetAttribute(gemv_kernel<MM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kSmemMax));
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ntile, nsplit, 1);
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = nsplit;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = nsplit > 1 ? 1 : 0;
  AWQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, gemv_kernel<MM>, X, qweight, scales, zeros, inv_s, N, K,
                                  KS, xs_stride, Y));
  return AWQ_OK;
}

}  // namespace

int launch_gemv(const __half* X, int M, const uint32_t* qweight, const __half* scales,
                const uint32_t* zeros, const float* inv_s, int N, int K, __half* Y,
                cudaStream_t st) {
  switch (M) {
    case 1: return launch_mm<1>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    case 2: return launch_mm<2>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    case 3: return launch_mm<3>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    case 4: return launch_mm<4>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    case 5: return launch_mm<5>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    case 6: return launch_mm<6>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    case 7: return launch_mm<7>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    case 8: return launch_mm<8>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    default: set_error("awq_gemv: M = %d must be in [1, 8]", M); return AWQ_ERR_SHAPE;
  }
}

}  // namespace awq
