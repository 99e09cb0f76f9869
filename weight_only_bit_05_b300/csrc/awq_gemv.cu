// W4A16 GEMV for M <= 8 tokens on CUDA cores.
//
// "awq-quantization（AWQ量化技术）Skill" page, section 主要功能和特点: a GEMV kernel
// serves batch-1 token generation; "AWQ量化实战" §3.4: decoding is bound by the
// bandwidth of reading the weights.  At the B300's HBM rate an SM must retire
// about 5.4 packed words (43 codes) per cycle, i.e. fewer than ~24 issue
// slots per word and ~12 integer-pipe operations per word, so the kernel is
// built around the instruction count per word:
//
//  * codes become exact fp32 numbers with ONE LOP3 per code: the nibble at
//    bit position p is OR-ed into the mantissa of 2^(23-p), giving
//    2^(23-p) + q (p = 0, 4, 8 of the word and of the word >> 12, the shift
//    done as a high multiply on the FMA pipe); four packed FADD2 remove the
//    constant offsets, four packed FFMA2 accumulate x~ * q in fp32 (exact
//    products of an fp32 activation and a 4-bit integer);
//  * the zero point and the step are applied once per half group (8 words):
//    y += s * (sum_k x~ q - z * sum_k x~), with the half-group sums of x~
//    precomputed in shared memory;
//  * a unit is R rows (4 at M = 1) x 16 groups: lane l reads 32 contiguous
//    bytes (half a group) of each row, every activation vector read from
//    shared memory serves R rows, and the next unit's codes are loaded into
//    registers while the current one is computed;
//  * one CTA per SM owns a balanced range of rows over the whole K; its warps
//    take units from a shared-memory counter, each unit's row sums are
//    reduced with warp shuffles into a per-(row, block) slot, and the slots
//    are added in a fixed order (deterministic whatever warp took a unit);
//  * only when the activations of a whole row do not fit in shared memory is
//    K split across the CTAs of a thread-block cluster, reduced in rank order
//    through distributed shared memory.
#include <cooperative_groups.h>

#include "awq_internal.h"

namespace cg = cooperative_groups;

namespace awq {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxSplit = 8;
constexpr int kGroupsPerUnit = 16;                 // 32 lanes x half a group
constexpr int kXsBudget = 160 * 1024;              // fp32 activation bytes per CTA

template <uint32_t MASK>
__device__ __forceinline__ float code_f32(uint32_t v, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(v), "n"(MASK), "r"(magic));
  return __uint_as_float(d);
}

struct Magic {
  uint32_t m23, m19, m15, m11, m7;   // bit patterns of 2^23, 2^19, 2^15, 2^11, 2^7
  float2 o01, o23, o45, o67;         // minus the offsets of codes (0,1) (2,3) (4,5) (6,7)
};

// acc += x~[k0..k7] * q[k0..k7] for the 8 codes of word w; hi = w >> 12.
__device__ __forceinline__ void word_dot(uint32_t w, uint32_t hi, const Magic& mg,
                                         const float4& xa, const float4& xb, float2& acc) {
  const float f0 = code_f32<0x0000000Fu>(w, mg.m23);    // 2^23 + q0
  const float f1 = code_f32<0x000000F0u>(w, mg.m19);    // 2^19 + q1
  const float f2 = code_f32<0x00000F00u>(w, mg.m15);    // 2^15 + q2
  const float f3 = code_f32<0x0000000Fu>(hi, mg.m23);   // 2^23 + q3
  const float f4 = code_f32<0x000000F0u>(hi, mg.m19);   // 2^19 + q4
  const float f5 = code_f32<0x00000F00u>(hi, mg.m15);   // 2^15 + q5
  const float f6 = code_f32<0x0000F000u>(hi, mg.m11);   // 2^11 + q6
  const float f7 = code_f32<0x000F0000u>(hi, mg.m7);    // 2^7  + q7
  const float2 q01 = __fadd2_rn(make_float2(f0, f1), mg.o01);
  const float2 q23 = __fadd2_rn(make_float2(f2, f3), mg.o23);
  const float2 q45 = __fadd2_rn(make_float2(f4, f5), mg.o45);
  const float2 q67 = __fadd2_rn(make_float2(f6, f7), mg.o67);
  acc = __ffma2_rn(make_float2(xa.x, xa.y), q01, acc);
  acc = __ffma2_rn(make_float2(xa.z, xa.w), q23, acc);
  acc = __ffma2_rn(make_float2(xb.x, xb.y), q45, acc);
  acc = __ffma2_rn(make_float2(xb.z, xb.w), q67, acc);
}

template <int MM, int R>
struct UnitRegs {
  uint4 w[R][2];      // 8 packed words of each row
  float s[R];         // group step
  float z[R];         // zero point
};

template <int MM, int R>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const __half* __restrict__ X, const uint32_t* __restrict__ qweight,
                const __half* __restrict__ scales, const uint32_t* __restrict__ zeros,
                const float* __restrict__ inv_s, int N, int K, int KS, int rows_cap,
                uint32_t hi_mult, __half* __restrict__ Y) {
  extern __shared__ float4 smem_f4[];
  __shared__ int next_unit;
  const int kbeg = blockIdx.y * KS;
  const int klen = min(K - kbeg, KS);              // multiple of 128
  const int Gs = klen / kGroup;
  // B: blocks of 16 groups in this slice; the shared-memory layout uses Bl,
  // the block count of a full slice, so that it is the same in every rank
  const int B = (Gs + kGroupsPerUnit - 1) / kGroupsPerUnit;
  const int Bl = (KS / kGroup + kGroupsPerUnit - 1) / kGroupsPerUnit;
  const int gbeg = kbeg / kGroup;
  float4* xs = smem_f4;                                       // [MM][Bl][8 words][2][32]
  float* xsum = reinterpret_cast<float*>(xs + static_cast<size_t>(MM) * Bl * 512);   // [MM][Bl][32]
  float* part = xsum + static_cast<size_t>(MM) * Bl * 32;     // [MM][rows_cap][Bl]

  // rows of this CTA: whole units of R rows, balanced over gridDim.x
  const int NU = N / R;
  const int q0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * NU / gridDim.x);
  const int q1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * NU / gridDim.x);
  const int row_base = q0 * R;
  const int nunits = (q1 - q0) * B;
  const int G = K / kGroup, ZW = (G + 7) / 8, KW = K / 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // unit u -> (row unit, block); lane -> half group
  auto issue = [&](int u, UnitRegs<MM, R>& ur) {
    const int qu = u / B, b = u - qu * B;
    const int gl = b * kGroupsPerUnit + (lane >> 1);
    if (gl < Gs) {
      const int g = gbeg + gl;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int row = row_base + qu * R + r;
        const uint4* src = reinterpret_cast<const uint4*>(qweight + static_cast<size_t>(row) * KW +
                                                          g * 16 + (lane & 1) * 8);
        ur.w[r][0] = __ldg(src);
        ur.w[r][1] = __ldg(src + 1);
        ur.s[r] = __half2float(scales[static_cast<size_t>(row) * G + g]);
        const uint32_t zw = __ldg(zeros + static_cast<size_t>(row) * ZW + (g >> 3));
        ur.z[r] = static_cast<float>((zw >> ((g & 7) * 4)) & 15u);
      }
    }
  };

  // the first unit's codes are requested before the activations are staged
  UnitRegs<MM, R> cur, nxt;
  int u = warp < nunits ? warp : nunits;
  if (u < nunits) issue(u, cur);
  if (threadIdx.x == 0) next_unit = kWarps;

  // ---- prologue: x~ = fp32(x) * inv_s into shared memory, half-group sums
  const int nw = klen / 8;
  for (int base = (threadIdx.x & ~31); base < MM * nw; base += kThreads) {
    const int idx = base + lane;
    const bool ok = idx < MM * nw;
    float f[8];
    float sum = 0.f;
    int m = 0, c = 0;
    if (ok) {
      m = idx / nw;
      c = idx - m * nw;
      const uint4 xr = __ldg(reinterpret_cast<const uint4*>(X + static_cast<size_t>(m) * K + kbeg + 8 * c));
      const __half2* xh = reinterpret_cast<const __half2*>(&xr);
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
#pragma unroll
      for (int i = 0; i < 8; ++i) sum += f[i];
      // word c: half group hg = c / 8 (lane of the unit = hg % 32), word j = c % 8
      const int hg = c >> 3, j = c & 7, b = hg >> 5, l = hg & 31;
      float4* dst = xs + ((static_cast<size_t>(m) * Bl + b) * 8 + j) * 64 + l;
      dst[0] = make_float4(f[0], f[1], f[2], f[3]);
      dst[32] = make_float4(f[4], f[5], f[6], f[7]);
    }
    // half-group sum over the 8 consecutive words (lanes 8i..8i+7)
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    if (ok && (c & 7) == 0) {
      const int hg = c >> 3;
      xsum[(static_cast<size_t>(m) * Bl + (hg >> 5)) * 32 + (hg & 31)] = sum;
    }
  }
  for (int i = threadIdx.x; i < MM * rows_cap * Bl; i += kThreads) part[i] = 0.f;
  __syncthreads();

  Magic mg;
  mg.m23 = 0x4B000000u;
  mg.m19 = 0x49000000u;
  mg.m15 = 0x47000000u;
  mg.m11 = 0x45000000u;
  mg.m7 = 0x43000000u;
  mg.o01 = make_float2(-8388608.f, -524288.f);
  mg.o23 = make_float2(-32768.f, -8388608.f);
  mg.o45 = make_float2(-524288.f, -32768.f);
  mg.o67 = make_float2(-2048.f, -128.f);

  // ---- main loop: dynamic units, next unit's codes in flight during compute
  while (u < nunits) {
    int un = 0;
    if (lane == 0) un = atomicAdd(&next_unit, 1);
    un = __shfl_sync(0xffffffffu, un, 0);
    if (un < nunits) issue(un, nxt);

    const int qu = u / B, b = u - qu * B;
    const int gl = b * kGroupsPerUnit + (lane >> 1);
    float res[R][MM];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MM; ++m) res[r][m] = 0.f;
    if (gl < Gs) {
#pragma unroll
      for (int m = 0; m < MM; ++m) {
        const float4* xp = xs + (static_cast<size_t>(m) * Bl + b) * 512 + lane;
        float2 acc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 xa = xp[j * 64];
          const float4 xb = xp[j * 64 + 32];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const uint4& q4 = cur.w[r][j >> 2];
            const uint32_t w = (j & 3) == 0 ? q4.x : (j & 3) == 1 ? q4.y : (j & 3) == 2 ? q4.z : q4.w;
            word_dot(w, __umulhi(w, hi_mult), mg, xa, xb, acc[r]);
          }
        }
        const float xsm = xsum[(static_cast<size_t>(m) * Bl + b) * 32 + lane];
#pragma unroll
        for (int r = 0; r < R; ++r) res[r][m] = cur.s[r] * ((acc[r].x + acc[r].y) - cur.z[r] * xsm);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MM; ++m) {
        float v = res[r][m];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) part[(static_cast<size_t>(m) * rows_cap + qu * R + r) * Bl + b] = v;
      }
    u = un;
    cur = nxt;
  }
  __syncthreads();

  // ---- fixed-order sums over the group blocks; cluster reduction over K slices
  const int nrows = (q1 - q0) * R;
  for (int i = threadIdx.x; i < MM * nrows; i += kThreads) {
    const int m = i / nrows, rl = i - m * nrows;
    const float* p = part + (static_cast<size_t>(m) * rows_cap + rl) * Bl;
    float v = 0.f;
    for (int b = 0; b < B; ++b) v += p[b];
    if (gridDim.y == 1)
      Y[static_cast<size_t>(m) * N + row_base + rl] = __float2half_rn(v);
    else
      part[(static_cast<size_t>(m) * rows_cap + rl) * Bl] = v;   // slot 0 holds the row total
  }
  if (gridDim.y == 1) return;
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  if (cluster.block_rank() == 0) {
    for (int i = threadIdx.x; i < MM * nrows; i += kThreads) {
      const int m = i / nrows, rl = i - m * nrows;
      const size_t slot = (static_cast<size_t>(m) * rows_cap + rl) * Bl;
      float v = 0.f;
      for (int rk = 0; rk < static_cast<int>(gridDim.y); ++rk)
        v += cluster.map_shared_rank(part, rk)[slot];
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
  constexpr int R = MM == 1 ? 4 : 1;
  const int G = K / kGroup;
  auto xs_bytes = [](int gs) {   // fp32 activations + half-group sums of one slice
    const int b = (gs + kGroupsPerUnit - 1) / kGroupsPerUnit;
    return static_cast<int64_t>(MM) * b * (512 * 16 + 32 * 4);
  };
  int nsplit = 1;
  while (nsplit < kMaxSplit && xs_bytes((G + nsplit - 1) / nsplit) > kXsBudget) ++nsplit;
  const int gs = (G + nsplit - 1) / nsplit;
  if (xs_bytes(gs) > kXsBudget) {
    set_error("awq_gemv: K = %d is too large for M = %d (use awq_gemm)", K, MM);
    return AWQ_ERR_SHAPE;
  }
  const int KS = gs * kGroup;
  nsplit = (K + KS - 1) / KS;
  const int B = (gs + kGroupsPerUnit - 1) / kGroupsPerUnit;
  const int units = N / R;
  int gx = num_sms() / nsplit;
  if (gx > units) gx = units;
  if (gx < 1) gx = 1;
  const int rows_cap = ((units + gx - 1) / gx) * R;
  const size_t smem = static_cast<size_t>(xs_bytes(gs)) +
                      static_cast<size_t>(MM) * rows_cap * B * sizeof(float);
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
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = nsplit;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = nsplit > 1 ? 1 : 0;
  // 2^20 as a run-time value: w * 2^20 >> 32 (= w >> 12) stays a high multiply
  // on the FMA pipe instead of becoming an integer-pipe shift
  const uint32_t hi_mult = 1u << 20;
  AWQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, gemv_kernel<MM, R>, X, qweight, scales, zeros, inv_s, N,
                                  K, KS, rows_cap, hi_mult, Y));
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
