// W4A16 GEMV for M <= 8 tokens on CUDA cores.
//
// "awq-quantization（AWQ量化技术）Skill" page, section 主要功能和特点: a GEMV kernel
// serves batch-1 token generation; "AWQ量化实战" §3.4: decoding is bound by the
// bandwidth of reading the weights.  The kernel streams the packed codes from
// HBM exactly once and hides the fixed cost of a launch behind that stream:
//
//  * each CTA owns a balanced range of rows over the whole K; the rows of a
//    range are contiguous in memory, so before anything else the CTA asks
//    for its whole range (codes, steps, zero points) to be brought into L2
//    with bulk prefetches.  The kernel is launched with programmatic stream
//    serialization, so this starts while the previous kernel on the stream
//    is still finishing; all loads proper come after griddepcontrol.wait
//    (and see what that kernel wrote: the prefetch fills only the coherent L2);
//  * a lane owns one whole group (16 words = 64 contiguous bytes, one step and
//    one zero point) of a row per unit; a warp's unit is 32 consecutive groups
//    of 2 rows, so each activation vector read from shared memory serves two
//    rows;
//  * the scaled activations x~ = fp16(fp32(x) * inv_s) are built once per CTA
//    into shared memory, interleaved so that the 32 lanes read 32 consecutive
//    16-byte vectors;
//  * codes become fp16 numbers with one LOP3 per pair: 1024 + q for the even
//    nibbles of a word and 64 + q for the odd nibbles (no shift needed for
//    half of them); HSUB2 of the matching (1024 + z) or (64 + z) gives q - z
//    exactly, and fma.rn.f32.f16 forms x~ (q - z) exactly in fp32 and adds it
//    to fp32 accumulators; the group step multiplies each group's sum;
//  * the 16 warps of a CTA split the CTA's (row pair, group block) units into
//    contiguous runs, flush a row's sum with warp shuffles into a per-warp
//    slot, and the slots are added in a fixed order (deterministic);
//  * only when the activations of the whole K do not fit in shared memory is
//    K split across the CTAs of a thread-block cluster, whose partial sums
//    are added in rank order through distributed shared memory.
#include <cooperative_groups.h>

#include "awq_internal.h"

namespace cg = cooperative_groups;

namespace awq {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxSplit = 8;
constexpr int kXsBudget = 96 * 1024;   // activation bytes per CTA (2 CTAs per SM)

__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(magic));
  return d;
}

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// c0 += a.lo * b.lo, c1 += a.hi * b.hi  (fp16 x fp16 exact, fp32 add)
__device__ __forceinline__ void fma_mixed2(uint32_t a, uint32_t b, float& c0, float& c1) {
  asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %2;\n mov.b32 {bl, bh}, %3;\n"
      " fma.rn.f32.f16 %0, al, bl, %0;\n fma.rn.f32.f16 %1, ah, bh, %1;\n}"
      : "+f"(c0), "+f"(c1)
      : "r"(a), "r"(b));
}

// x~ (q - z) for the 8 codes of one word into four fp32 accumulators.
// x holds the activations as fp16 pairs (k0,k4) (k1,k5) (k2,k6) (k3,k7).
__device__ __forceinline__ void word_dot(uint32_t w, uint32_t zb_even, uint32_t zb_odd,
                                         const uint4& x, float (&c)[4]) {
  const uint32_t t = w >> 8;
  const uint32_t d0 = hsub2_u(and_or(w, 0x000F000Fu, 0x64006400u), zb_even);   // (k0, k4)
  const uint32_t d1 = hsub2_u(and_or(w, 0x00F000F0u, 0x54005400u), zb_odd);    // (k1, k5)
  const uint32_t d2 = hsub2_u(and_or(t, 0x000F000Fu, 0x64006400u), zb_even);   // (k2, k6)
  const uint32_t d3 = hsub2_u(and_or(t, 0x00F000F0u, 0x54005400u), zb_odd);    // (k3, k7)
  fma_mixed2(d0, x.x, c[0], c[1]);
  fma_mixed2(d1, x.y, c[2], c[3]);
  fma_mixed2(d2, x.z, c[0], c[1]);
  fma_mixed2(d3, x.w, c[2], c[3]);
}

// Bulk L2 prefetch of [p, p + bytes) in pieces of at most 64 KB, spread over
// the lanes of the calling warp.
__device__ __forceinline__ void prefetch_range(const void* p, size_t bytes, int lane) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(p) & ~static_cast<uintptr_t>(15);
  const uintptr_t a1 = (reinterpret_cast<uintptr_t>(p) + bytes + 15) & ~static_cast<uintptr_t>(15);
  constexpr uintptr_t kPiece = 65536;
  for (uintptr_t a = a0 + lane * kPiece; a < a1; a += 32 * kPiece) {
    const uintptr_t e = a + kPiece < a1 ? a + kPiece : a1;
    prefetch_l2_bulk(reinterpret_cast<const void*>(a), static_cast<uint32_t>(e - a));
  }
}

template <int MM, int R>
__global__ void __launch_bounds__(kThreads, (MM <= 3 ? 2 : 1))
    gemv_kernel(const __half* __restrict__ X, const uint32_t* __restrict__ qweight,
                const __half* __restrict__ scales, const uint32_t* __restrict__ zeros,
                const float* __restrict__ inv_s, int N, int K, int KS, int rows_cap,
                __half* __restrict__ Y) {
  extern __shared__ uint4 smem_u4[];
  const int kbeg = blockIdx.y * KS;
  const int klen = min(K - kbeg, KS);          // multiple of 128
  const int Gs = klen / kGroup;                // groups in the slice
  const int B = (Gs + 31) / 32;                // group blocks of 32 (one per lane)
  const int gbeg = kbeg / kGroup;
  uint4* xs = smem_u4;                         // [MM][B*16][32]
  float* red = reinterpret_cast<float*>(xs + static_cast<size_t>(MM) * B * 512);   // [MM][kWarps][rows_cap]

  // rows of this CTA (whole units of R rows, balanced over gridDim.x)
  const int NU = N / R;
  const int u0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * NU / gridDim.x);
  const int u1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * NU / gridDim.x);
  const int row_base = u0 * R;
  const int nrows = (u1 - u0) * R;
  const int G = K / kGroup, ZW = (G + 7) / 8, KW = K / 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- start streaming this CTA's rows into L2 (before the dependency wait)
  if (warp == 0) {
    prefetch_range(qweight + static_cast<size_t>(row_base) * KW, static_cast<size_t>(nrows) * KW * 4, lane);
  } else if (warp == 1) {
    prefetch_range(scales + static_cast<size_t>(row_base) * G, static_cast<size_t>(nrows) * G * 2, lane);
    prefetch_range(zeros + static_cast<size_t>(row_base) * ZW, static_cast<size_t>(nrows) * ZW * 4, lane);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  // ---- prologue: x~ into shared memory, zero the per-warp row slots
  const int nw = klen / 8;   // packed words per row in the slice
  for (int idx = threadIdx.x; idx < MM * nw; idx += kThreads) {
    const int m = idx / nw, c = idx - m * nw;
    const int gl = c >> 4, j = c & 15, b = gl >> 5, l = gl & 31;
    const size_t xo = static_cast<size_t>(m) * K + kbeg + 8 * c;
    const uint4 xr = __ldg(reinterpret_cast<const uint4*>(X + xo));
    const __half2* xh = reinterpret_cast<const __half2*>(&xr);
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v = __half22float2(xh[i]);
      f[2 * i] = v.x;
      f[2 * i + 1] = v.y;
    }
    if (inv_s) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(inv_s + kbeg + 8 * c));
      const float4 bq = __ldg(reinterpret_cast<const float4*>(inv_s + kbeg + 8 * c + 4));
      const float is[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(f[i], is[i]);
    }
    uint4 o;
    __half2 p;
    p = __halves2half2(__float2half_rn(f[0]), __float2half_rn(f[4])); o.x = *reinterpret_cast<uint32_t*>(&p);
    p = __halves2half2(__float2half_rn(f[1]), __float2half_rn(f[5])); o.y = *reinterpret_cast<uint32_t*>(&p);
    p = __halves2half2(__float2half_rn(f[2]), __float2half_rn(f[6])); o.z = *reinterpret_cast<uint32_t*>(&p);
    p = __halves2half2(__float2half_rn(f[3]), __float2half_rn(f[7])); o.w = *reinterpret_cast<uint32_t*>(&p);
    xs[(static_cast<size_t>(m) * B + b) * 512 + j * 32 + l] = o;
  }
  for (int i = threadIdx.x; i < MM * kWarps * rows_cap; i += kThreads) red[i] = 0.f;
  __syncthreads();

  // ---- main loop over this warp's contiguous run of (row unit, group block)
  const int nunits = (u1 - u0) * B;
  const int ub = static_cast<int>(static_cast<int64_t>(warp) * nunits / kWarps);
  const int ue = static_cast<int>(static_cast<int64_t>(warp + 1) * nunits / kWarps);

  float acc[R][MM];
  int cur = -1;
  auto flush = [&](int unit_row) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MM; ++m) {
        float v = acc[r][m];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) red[(m * kWarps + warp) * rows_cap + unit_row * R + r] = v;
      }
  };

  for (int u = ub; u < ue; ++u) {
    const int ul = u / B, b = u - ul * B;
    if (ul != cur) {
      if (cur >= 0) flush(cur);
      cur = ul;
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MM; ++m) acc[r][m] = 0.f;
    }
    const int gl = b * 32 + lane;
    if (gl < Gs) {
      const int g = gbeg + gl;
      uint4 wq[R][4];
      float s[R];
      uint32_t zbe[R], zbo[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int row = row_base + ul * R + r;
        const uint4* src = reinterpret_cast<const uint4*>(qweight + static_cast<size_t>(row) * KW + g * 16);
#pragma unroll
        for (int v = 0; v < 4; ++v) wq[r][v] = __ldg(src + v);
        s[r] = __half2float(scales[static_cast<size_t>(row) * G + g]);
        const uint32_t z = (__ldg(zeros + static_cast<size_t>(row) * ZW + (g >> 3)) >> ((g & 7) * 4)) & 15u;
        zbe[r] = (0x6400u | z) * 0x00010001u;          // (1024 + z, 1024 + z)
        zbo[r] = (0x5400u | (z << 4)) * 0x00010001u;   // (64 + z, 64 + z)
      }
      float c[R][MM][4];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MM; ++m)
#pragma unroll
          for (int i = 0; i < 4; ++i) c[r][m][i] = 0.f;
      const uint4* xp = xs + static_cast<size_t>(b) * 512 + lane;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
#pragma unroll
        for (int m = 0; m < MM; ++m) {
          const uint4 xv = xp[static_cast<size_t>(m) * B * 512 + j * 32];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const uint4& q4 = wq[r][j >> 2];
            const uint32_t w = (j & 3) == 0 ? q4.x : (j & 3) == 1 ? q4.y : (j & 3) == 2 ? q4.z : q4.w;
            word_dot(w, zbe[r], zbo[r], xv, c[r][m]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MM; ++m)
          acc[r][m] = fmaf(s[r], (c[r][m][0] + c[r][m][1]) + (c[r][m][2] + c[r][m][3]), acc[r][m]);
    }
  }
  if (cur >= 0) flush(cur);
  __syncthreads();

  // ---- fixed-order sum of the per-warp slots; cluster reduction over K slices
  float* total = red;   // warp 0's slots hold the CTA total in the cluster case
  for (int i = threadIdx.x; i < MM * nrows; i += kThreads) {
    const int m = i / nrows, rl = i - m * nrows;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v += red[(m * kWarps + w) * rows_cap + rl];
    if (gridDim.y == 1)
      Y[static_cast<size_t>(m) * N + row_base + rl] = __float2half_rn(v);
    else
      total[m * kWarps * rows_cap + rl] = v;   // only the slot read by this thread changes
  }
  if (gridDim.y == 1) return;
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  if (cluster.block_rank() == 0) {
    for (int i = threadIdx.x; i < MM * nrows; i += kThreads) {
      const int m = i / nrows, rl = i - m * nrows;
      float v = 0.f;
      for (int rk = 0; rk < static_cast<int>(gridDim.y); ++rk)
        v += cluster.map_shared_rank(total, rk)[m * kWarps * rows_cap + rl];
      Y[static_cast<size_t>(m) * N + row_base + rl] = __float2half_rn(v);
    }
  }
  cluster.sync();   // every CTA's shared memory stays alive until rank 0 has read it
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
  constexpr int R = MM <= 2 ? 2 : 1;
  const int G = K / kGroup;
  // K slices: activations of a slice take MM * 8 KB per 32 groups; split K
  // only when the whole row does not fit the budget
  int nsplit = 1;
  while (nsplit < kMaxSplit &&
         static_cast<int64_t>(MM) * (((G + nsplit - 1) / nsplit + 31) / 32) * 8192 > kXsBudget)
    ++nsplit;
  const int gs = (G + nsplit - 1) / nsplit;
  if (static_cast<int64_t>(MM) * ((gs + 31) / 32) * 8192 > 200 * 1024) {
    set_error("awq_gemv: K = %d is too large for M = %d (use awq_gemm)", K, MM);
    return AWQ_ERR_SHAPE;
  }
  const int KS = gs * kGroup;
  nsplit = (K + KS - 1) / KS;
  const int B = (gs + 31) / 32;
  const int units = N / R;
  int gx = 2 * num_sms() / nsplit;
  if (gx > units) gx = units;
  if (gx < 1) gx = 1;
  const int rows_cap = ((units + gx - 1) / gx) * R;
  const size_t smem = static_cast<size_t>(MM) * B * 512 * sizeof(uint4) +
                      static_cast<size_t>(MM) * kWarps * rows_cap * sizeof(float);
  if (smem > 220 * 1024) {
    set_error("awq_gemv: shared memory plan of %zu bytes too large (N = %d, K = %d, M = %d)",
              smem, N, K, MM);
    return AWQ_ERR_SHAPE;
  }
  static bool attr_set = false;
  if (!attr_set) {
    AWQ_CUDA_TRY(cudaFuncSetAttribute(gemv_kernel<MM, R>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024));
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gx, nsplit, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = nsplit;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = nsplit > 1 ? 2 : 1;
  AWQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, gemv_kernel<MM, R>, X, qweight, scales, zeros, inv_s, N,
                                  K, KS, rows_cap, Y));
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
