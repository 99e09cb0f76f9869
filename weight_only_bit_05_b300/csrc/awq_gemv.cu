// W4A16 GEMV for M <= 8 tokens on CUDA cores.
//
// "awq-quantization（AWQ量化技术）Skill" page, section 主要功能和特点: a GEMV kernel
// serves batch-1 token generation; "AWQ量化实战" §3.4: decoding is bound by the
// bandwidth of reading the weights.  The kernel streams the packed codes from
// HBM exactly once.  On B300 a single token leaves it bound by the issue rate
// of the dequantize-and-multiply instructions (about 23 per packed word) on
// large layers and by the fixed latency of a launch on small ones:
//
//  * each CTA owns a balanced range of rows over the whole K, one CTA per SM;
//    the rows of a range are contiguous in memory.  The kernel is launched
//    with programmatic stream serialization.  Before griddepcontrol.wait a CTA
//    asks for the head of its range (at most 128 KB of codes, with its steps
//    and zero points) to be brought into L2 with bulk prefetches.  They fill
//    only the coherent L2, so they are safe while the previous kernel is still
//    writing.  The head is bounded because prefetching a whole large layer at
//    once evicts lines before they are read;
//  * a lane owns one whole group (16 words = 64 contiguous bytes, one step and
//    one zero point) of a row per unit; a warp's unit is 32 consecutive groups
//    of R rows (R = 2 for M <= 2), so each activation vector read from shared
//    memory serves R rows;
//  * the scaled activations x~ = fp16(fp32(x) * inv_s) are built once per CTA
//    into shared memory, interleaved so that the 32 lanes read 32 consecutive
//    16-byte vectors;
//  * codes become fp16 numbers with one LOP3 per pair: 1024 + q for the even
//    nibbles of a word and 64 + q for the odd nibbles (no shift needed for
//    half of them); HSUB2 of the matching (1024 + z) or (64 + z) gives q - z
//    exactly, and fma.rn.f32.f16 forms x~ (q - z) exactly in fp32 and adds it
//    to fp32 accumulators; the group step multiplies each group's sum;
//  * the warps of a CTA split the CTA's (row unit, group block) units into
//    contiguous runs and reduce a row's sum over the lanes with warp
//    shuffles.  For one or two tokens each warp writes its own slot per row
//    and the slots are added in warp order; for more tokens a row unit owned
//    by one warp is written to the CTA's row totals at once and a unit split
//    between neighbouring warps is finished after one barrier by adding their
//    partial sums in warp order.  Both are deterministic, and the totals leave
//    shared memory as coalesced fp16 stores;
//  * launch shapes: 32 warps (64 registers each) for one or two tokens; 16
//    warps that take half an SM for the smallest layers, so the next GEMV's
//    CTA can already sit on the SM and run its prefetch; 16 warps with 128
//    registers for 3 to 8 tokens, whose accumulators need them;
//  * only when the activations of the whole K do not fit in shared memory is
//    K split across the CTAs of a thread-block cluster, whose partial sums
//    are added in rank order through distributed shared memory.
#include <cooperative_groups.h>

#include "awq_internal.h"

namespace cg = cooperative_groups;

namespace awq {
namespace {

constexpr int kMaxSplit = 8;
constexpr size_t kHeadPrefetch = 128 * 1024;   // codes per CTA prefetched into L2 before the wait
// Layers with at most this many bytes of codes per SM run the 16-warp CTA that
// leaves room for the next kernel's CTA on the same SM (one or two tokens).
constexpr size_t kSmallBytesPerSm = 64 * 1024;

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

// x~ (q - z) for the 4 codes of one 8-bit word into four fp32 accumulators:
// bytes 0 and 2 (bits 0..7 of each half) and bytes 1 and 3 become 1024 + q;
// xa holds the activations (k0, k2), xb (k1, k3).
__device__ __forceinline__ void word_dot8(uint32_t w, uint32_t zb, uint32_t xa, uint32_t xb,
                                          float (&c)[4]) {
  const uint32_t d0 = hsub2_u(and_or(w, 0x00FF00FFu, 0x64006400u), zb);        // (k0, k2)
  const uint32_t d1 = hsub2_u(and_or(w >> 8, 0x00FF00FFu, 0x64006400u), zb);   // (k1, k3)
  fma_mixed2(d0, xa, c[0], c[1]);
  fma_mixed2(d1, xb, c[2], c[3]);
}

// MM tokens, R rows per unit, kWarps warps per CTA, MINB CTAs per SM for the
// register budget.  SILU: the weight stacks I gate rows over I up rows and the
// kernel writes silu(gate) * up ([M][I]); it walks "virtual" rows v in which
// v = 2j is gate row j and v = 2j + 1 up row j, so a row unit of R = 2 holds
// one (gate, up) pair and a CTA's range always holds whole pairs.
// BITS-bit codes (4 or 8) with GS-channel groups (128, 64 or 32): a lane
// chunk is always 16 packed words (128 channels of 4-bit codes, 64 of 8-bit);
// groups smaller than a chunk are segments with their own step and zero
// point, folded into the row sum as each segment ends.
template <int MM, int R, int kWarps, int MINB, bool SILU, int BITS, int GS>
__global__ void __launch_bounds__(kWarps * 32, MINB)
    gemv_kernel(const __half* __restrict__ X, const uint32_t* __restrict__ qweight,
                const __half* __restrict__ scales, const uint32_t* __restrict__ zeros,
                const float* __restrict__ inv_s, int N, int K, int KS, int rows_cap,
                __half* __restrict__ Y) {
  constexpr int kThreads = kWarps * 32;
  constexpr int CK = BITS == 4 ? 128 : 64;      // input channels per lane chunk
  constexpr int OCT = CK / 8;                   // x~ vectors (8 channels) per chunk
  constexpr int XB = 32 * OCT;                  // x~ vectors per block of 32 chunks
  constexpr int NSEG = CK > GS ? CK / GS : 1;   // groups per chunk
  constexpr int SEGW = 16 / NSEG;               // packed words per group segment
  constexpr int PW = 32 / BITS;                 // codes per packed word
  constexpr uint32_t QMASK = (1u << BITS) - 1u;
  extern __shared__ uint4 smem_u4[];
  const int kbeg = blockIdx.y * KS;
  const int klen = min(K - kbeg, KS);          // multiple of 128
  const int Cs = klen / CK;                    // lane chunks in the slice
  const int B = (Cs + 31) / 32;                // chunk blocks of 32 (one chunk per lane)
  const int cbeg = kbeg / CK;
  uint4* xs = smem_u4;                         // [MM][B][OCT][32]
  // Row sums.  For one or two tokens every warp has its own slot per row,
  // red[MM][kWarps][rows_cap], added in warp order at the end; for more tokens
  // (where that table would not fit) a row unit owned by one warp goes to
  // tot[MM][rows_cap] at once and the units split between warps meet in
  // part[kWarps][2][R*MM].
  constexpr bool kSlots = MM <= 2;
  float* red = reinterpret_cast<float*>(xs + static_cast<size_t>(MM) * B * XB);
  float* tot = red;
  float* part = tot + MM * rows_cap;
  constexpr int kTotStride = kSlots ? kWarps : 1;   // tot[m][rl] sits at red[m][0][rl] then

  // rows of this CTA (whole units of R rows, or whole (gate, up) pairs,
  // balanced over gridDim.x)
  const int NB = SILU ? N / 2 : N / R;
  const int per = SILU ? 2 / R : 1;    // row units per balancing unit
  const int u0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * NB / gridDim.x) * per;
  const int u1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * NB / gridDim.x) * per;
  const int row_base = u0 * R;         // first (virtual) row of the CTA
  const int half_n = N >> 1;
  // physical row of virtual row v
  auto phys = [&](int v) { return SILU ? (v >> 1) + (v & 1) * half_n : v; };
  const int nrows = (u1 - u0) * R;
  const int G = K / GS, ZW = (G + PW - 1) / PW, KW = K / PW;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- the head of this CTA's rows into L2, before the dependency wait
  if (warp == 0 && gridDim.y == 1) {
    // one contiguous physical range, or the gate and the up range
    constexpr int kRanges = SILU ? 2 : 1;
    const int prow = SILU ? nrows / 2 : nrows;
    constexpr size_t cap = kHeadPrefetch / kRanges;
    for (int h = 0; h < kRanges; ++h) {
      const size_t r0 = static_cast<size_t>(phys(row_base + h));
      const size_t qb = static_cast<size_t>(prow) * KW * 4;
      const size_t sb = static_cast<size_t>(prow) * G * 2;
      const size_t zb = static_cast<size_t>(prow) * ZW * 4;
      prefetch_range(qweight + r0 * KW, qb < cap ? qb : cap, lane);
      prefetch_range(scales + r0 * G, sb < cap / 32 ? sb : cap / 32, lane);
      prefetch_range(zeros + r0 * ZW, zb < cap / 128 ? zb : cap / 128, lane);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  // ---- prologue: x~ into shared memory, zero the per-warp row slots.  An
  // 8-channel vector holds the fp16 pairs (k0,k4) (k1,k5) (k2,k6) (k3,k7) for
  // 4-bit codes (one packed word) and (k0,k2) (k1,k3) (k4,k6) (k5,k7) for
  // 8-bit codes (two packed words), the pairs the dequantization produces.
  const int n8 = klen / 8;   // 8-channel vectors per row in the slice
  for (int idx = threadIdx.x; idx < MM * n8; idx += kThreads) {
    const int m = idx / n8, c = idx - m * n8;
    const int cl = c / OCT, o = c - cl * OCT, b = cl >> 5, l = cl & 31;
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
    // pair partners: i and i + 4 (4-bit), or within each half i and i + 2
    constexpr int lo[4] = {0, 1, BITS == 4 ? 2 : 4, BITS == 4 ? 3 : 5};
    constexpr int step = BITS == 4 ? 4 : 2;
    uint4 o4;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o4);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 p = __halves2half2(__float2half_rn(f[lo[i]]), __float2half_rn(f[lo[i] + step]));
      ow[i] = *reinterpret_cast<const uint32_t*>(&p);
    }
    xs[(static_cast<size_t>(m) * B + b) * XB + o * 32 + l] = o4;
  }
  if (kSlots)
    for (int i = threadIdx.x; i < MM * kWarps * rows_cap; i += kThreads) red[i] = 0.f;
  __syncthreads();

  // ---- main loop over this warp's contiguous run [ub, ue) of (row unit,
  // group block) pairs.  Without per-warp slots, a row unit whose blocks all
  // lie in the run has its total written to tot at once, and the partial sums
  // of a unit split between neighbouring warps go to part (slot 0: the run's
  // first row unit, slot 1: its last) and are added after the loop.
  constexpr int RM = R * MM;
  const int nunits = (u1 - u0) * B;
  const int ub = static_cast<int>(static_cast<int64_t>(warp) * nunits / kWarps);
  const int ue = static_cast<int>(static_cast<int64_t>(warp + 1) * nunits / kWarps);
  const int ul_first = ub / B;

  float acc[R][MM];
  int cur = -1;
  auto flush = [&](int unit_row) {
    const bool whole = unit_row * B >= ub && (unit_row + 1) * B <= ue;
    const int slot = unit_row == ul_first ? 0 : 1;
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MM; ++m) {
        float v = acc[r][m];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) {
          if (kSlots)
            red[(m * kWarps + warp) * rows_cap + unit_row * R + r] = v;
          else if (whole)
            tot[m * rows_cap + unit_row * R + r] = v;
          else
            part[(warp * 2 + slot) * RM + r * MM + m] = v;
        }
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
    const int cl = b * 32 + lane;
    if (cl < Cs) {
      const int c = cbeg + cl;                  // chunk index in the row
      const int g0 = c * CK / GS;               // group of the chunk's first segment
      uint4 wq[R][4];
      float s[R][NSEG];
      uint32_t zbe[R][NSEG], zbo[R][NSEG];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int row = phys(row_base + ul * R + r);
        const uint4* src = reinterpret_cast<const uint4*>(qweight + static_cast<size_t>(row) * KW + c * 16);
#pragma unroll
        for (int v = 0; v < 4; ++v) wq[r][v] = __ldg(src + v);
#pragma unroll
        for (int sg = 0; sg < NSEG; ++sg) {
          const int g = g0 + sg;
          s[r][sg] = __half2float(scales[static_cast<size_t>(row) * G + g]);
          const uint32_t z =
              (__ldg(zeros + static_cast<size_t>(row) * ZW + g / PW) >> ((g % PW) * BITS)) & QMASK;
          zbe[r][sg] = (0x6400u | z) * 0x00010001u;          // (1024 + z, 1024 + z)
          zbo[r][sg] = (0x5400u | (z << 4)) * 0x00010001u;   // (64 + z, 64 + z), 4-bit only
        }
      }
      float c4[R][MM][4];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MM; ++m)
#pragma unroll
          for (int i = 0; i < 4; ++i) c4[r][m][i] = 0.f;
      // a finished segment: its step times its sum joins the row sum
      auto fold = [&](int sg) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int m = 0; m < MM; ++m) {
            acc[r][m] = fmaf(s[r][sg], (c4[r][m][0] + c4[r][m][1]) + (c4[r][m][2] + c4[r][m][3]),
                             acc[r][m]);
#pragma unroll
            for (int i = 0; i < 4; ++i) c4[r][m][i] = 0.f;
          }
      };
      const uint4* xp = xs + static_cast<size_t>(b) * XB + lane;
      auto word = [&](int r, int j) {
        const uint4& q4 = wq[r][j >> 2];
        return (j & 3) == 0 ? q4.x : (j & 3) == 1 ? q4.y : (j & 3) == 2 ? q4.z : q4.w;
      };
      if constexpr (BITS == 4) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
#pragma unroll
          for (int m = 0; m < MM; ++m) {
            const uint4 xv = xp[static_cast<size_t>(m) * B * XB + j * 32];
#pragma unroll
            for (int r = 0; r < R; ++r)
              word_dot(word(r, j), zbe[r][j / SEGW], zbo[r][j / SEGW], xv, c4[r][m]);
          }
          if (j % SEGW == SEGW - 1) fold(j / SEGW);
        }
      } else {
#pragma unroll
        for (int o = 0; o < 8; ++o) {
#pragma unroll
          for (int m = 0; m < MM; ++m) {
            const uint4 xv = xp[static_cast<size_t>(m) * B * XB + o * 32];
#pragma unroll
            for (int r = 0; r < R; ++r) {
              word_dot8(word(r, 2 * o), zbe[r][(2 * o) / SEGW], xv.x, xv.y, c4[r][m]);
              word_dot8(word(r, 2 * o + 1), zbe[r][(2 * o) / SEGW], xv.z, xv.w, c4[r][m]);
            }
          }
          if ((2 * o + 1) % SEGW == SEGW - 1) fold((2 * o) / SEGW);
        }
      }
    }
  }
  if (cur >= 0) flush(cur);
  __syncthreads();

  // outputs: one per row, or one per (gate, up) pair
  const int rstep = SILU ? 2 : 1;
  const int nout = nrows / rstep;
  const int ld_y = N / rstep;
  __half* yb = Y + row_base / rstep;
  auto put = [&](int m, int o, float a, float b) {
    const float y = SILU ? a / (1.f + expf(-a)) * b : a;
    yb[static_cast<size_t>(m) * ld_y + o] = __float2half_rn(y);
  };

  if (kSlots) {
    // fixed-order sum of the per-warp slots into warp 0's slot
    for (int i = threadIdx.x; i < MM * nout; i += kThreads) {
      const int m = i / nout, o = i - m * nout;
      float a = 0.f, b = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        a += red[(m * kWarps + w) * rows_cap + o * rstep];
        if (SILU) b += red[(m * kWarps + w) * rows_cap + o * rstep + 1];
      }
      if (gridDim.y == 1) {
        put(m, o, a, b);
      } else {   // only the slots read by this thread change
        red[m * kWarps * rows_cap + o * rstep] = a;
        if (SILU) red[m * kWarps * rows_cap + o * rstep + 1] = b;
      }
    }
    if (gridDim.y == 1) return;
  } else {
    // row units split between warps: the warp in whose run a unit starts
    // adds its own partial and those of the following warps, in warp order
    if (ub < ue && lane < RM) {
      const int ul_last = (ue - 1) / B;
      if (ul_last * B >= ub && (ul_last + 1) * B > ue) {
        const int r = lane / MM, m = lane - r * MM;
        float v = part[(warp * 2 + (ul_last == ul_first ? 0 : 1)) * RM + lane];
        const int stop = (ul_last + 1) * B;
        for (int w2 = warp + 1; w2 < kWarps; ++w2) {
          const int ub2 = static_cast<int>(static_cast<int64_t>(w2) * nunits / kWarps);
          const int ue2 = static_cast<int>(static_cast<int64_t>(w2 + 1) * nunits / kWarps);
          if (ub2 >= stop) break;
          if (ub2 < ue2) v += part[w2 * 2 * RM + lane];
        }
        tot[m * rows_cap + ul_last * R + r] = v;
      }
    }
    __syncthreads();
    if (gridDim.y == 1) {
      for (int i = threadIdx.x; i < MM * nout; i += kThreads) {
        const int m = i / nout, o = i - m * nout;
        put(m, o, tot[m * rows_cap + o * rstep], SILU ? tot[m * rows_cap + o * rstep + 1] : 0.f);
      }
      return;
    }
  }

  // ---- K split over a cluster: rank 0 adds the CTA totals in rank order
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  if (cluster.block_rank() == 0) {
    for (int i = threadIdx.x; i < MM * nout; i += kThreads) {
      const int m = i / nout, o = i - m * nout;
      float a = 0.f, b = 0.f;
      for (int rk = 0; rk < static_cast<int>(gridDim.y); ++rk) {
        const float* t = cluster.map_shared_rank(tot, rk) + m * kTotStride * rows_cap + o * rstep;
        a += t[0];
        if (SILU) b += t[1];
      }
      put(m, o, a, b);
    }
  }
  cluster.sync();   // every CTA's shared memory stays alive until rank 0 has read it
}

template <int MM, int R, int kWarps, int MINB, bool SILU, int BITS, int GS>
int launch_shape(const __half* X, const uint32_t* qweight, const __half* scales,
                 const uint32_t* zeros, const float* inv_s, int N, int K, __half* Y,
                 cudaStream_t st) {
  constexpr int CK = BITS == 4 ? 128 : 64;
  constexpr int XB = 32 * (CK / 8);
  // activation bytes a CTA may hold: a quarter of an SM's shared memory for
  // the half-SM shape, most of it otherwise
  constexpr int64_t kXsBudget = MINB == 2 ? 64 * 1024 : 160 * 1024;
  const int K128 = K / 128;
  // K slices, in whole 128-channel units: the activations of a slice take
  // MM * XB * 16 bytes per block of 32 lane chunks; split K only when the
  // whole row does not fit the budget
  auto xs_bytes = [&](int ns) {
    const int chunks = ((K128 + ns - 1) / ns) * (128 / CK);
    return static_cast<int64_t>(MM) * ((chunks + 31) / 32) * XB * 16;
  };
  int nsplit = 1;
  while (nsplit < kMaxSplit && xs_bytes(nsplit) > kXsBudget) ++nsplit;
  const int ks = (K128 + nsplit - 1) / nsplit;
  const int KS = ks * 128;
  nsplit = (K + KS - 1) / KS;
  const int B = (ks * (128 / CK) + 31) / 32;
  // balancing units: row units, or (gate, up) pairs
  const int units = SILU ? N / 2 : N / R;
  int gx = sm_count() / nsplit;
  if (gx > units) gx = units;
  if (gx < 1) gx = 1;
  const int rows_cap = ((units + gx - 1) / gx) * (SILU ? 2 : R);
  const size_t smem = static_cast<size_t>(MM) * B * XB * sizeof(uint4) +
                      (MM <= 2 ? static_cast<size_t>(MM) * kWarps * rows_cap * sizeof(float)
                               : static_cast<size_t>(MM) * rows_cap * sizeof(float) +
                                     static_cast<size_t>(kWarps) * 2 * R * MM * sizeof(float));
  if (smem > 220 * 1024) {
    set_error("awq_gemv: shared memory plan of %zu bytes too large (N = %d, K = %d, M = %d; "
              "use awq_gemm)", smem, N, K, MM);
    return AWQ_ERR_SHAPE;
  }
  auto kern = gemv_kernel<MM, R, kWarps, MINB, SILU, BITS, GS>;
  {
    const int rc = ensure_smem_attr(reinterpret_cast<const void*>(kern), 220 * 1024);
    if (rc != AWQ_OK) return rc;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gx, nsplit, 1);
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
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
  AWQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, X, qweight, scales, zeros, inv_s, N, K, KS,
                                  rows_cap, Y));
  return AWQ_OK;
}

template <int MM, bool SILU, int BITS, int GS>
int launch_mm(const __half* X, const uint32_t* qweight, const __half* scales,
              const uint32_t* zeros, const float* inv_s, int N, int K, __half* Y,
              cudaStream_t st) {
  if constexpr (MM <= 2) {
    // the half-SM shape for the smallest layers of the default format only
    constexpr bool kDefault = BITS == 4 && GS == 128;
    const size_t code_bytes = static_cast<size_t>(N) * K * BITS / 8;
    if (kDefault && code_bytes <= kSmallBytesPerSm * sm_count())
      return launch_shape<MM, 2, 16, 2, SILU, BITS, GS>(X, qweight, scales, zeros, inv_s, N, K,
                                                        Y, st);
    return launch_shape<MM, 2, 32, 1, SILU, BITS, GS>(X, qweight, scales, zeros, inv_s, N, K, Y,
                                                      st);
  } else {
    return launch_shape<MM, 1, 16, 1, SILU, BITS, GS>(X, qweight, scales, zeros, inv_s, N, K, Y,
                                                      st);
  }
}

template <bool SILU, int BITS, int GS>
int launch_m(const __half* X, int M, const uint32_t* qweight, const __half* scales,
             const uint32_t* zeros, const float* inv_s, int N, int K, __half* Y, cudaStream_t st) {
  switch (M) {
    case 1: return launch_mm<1, SILU, BITS, GS>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    case 2: return launch_mm<2, SILU, BITS, GS>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    case 3: return launch_mm<3, SILU, BITS, GS>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    case 4: return launch_mm<4, SILU, BITS, GS>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    case 5: return launch_mm<5, SILU, BITS, GS>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    case 6: return launch_mm<6, SILU, BITS, GS>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    case 7: return launch_mm<7, SILU, BITS, GS>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    case 8: return launch_mm<8, SILU, BITS, GS>(X, qweight, scales, zeros, inv_s, N, K, Y, st);
    default: set_error("awq_gemv: M = %d must be in [1, 8]", M); return AWQ_ERR_SHAPE;
  }
}

}  // namespace

int launch_gemv(const __half* X, int M, const uint32_t* qweight, const __half* scales,
                const uint32_t* zeros, const float* inv_s, int N, int K, __half* Y,
                cudaStream_t st, bool silu_mul, int w_bit, int group) {
  if (silu_mul) {
    if (w_bit != 4 || group != 128) {
      set_error("the fused gate/up layer takes 4-bit codes with 128-channel groups");
      return AWQ_ERR_UNSUPPORTED;
    }
    return launch_m<true, 4, 128>(X, M, qweight, scales, zeros, inv_s, N, K, Y, st);
  }
  if (gemv_mma_eligible(M, K, w_bit, group, false)) {
    const MmaGemvPlan p = plan_gemv_mma(M, N, K, sm_count());
    if (p.depth > 0)
      return launch_gemv_mma_plan(p, X, M, qweight, scales, zeros, inv_s, N, K, Y, st);
    // no shared-memory plan (many tokens on the largest layers): CUDA cores
  }
#define AWQ_GEMV_CASE(B, GS)                                                              \
  if (w_bit == B && group == GS)                                                          \
    return launch_m<false, B, GS>(X, M, qweight, scales, zeros, inv_s, N, K, Y, st);
  AWQ_GEMV_CASE(4, 128)
  AWQ_GEMV_CASE(4, 64)
  AWQ_GEMV_CASE(4, 32)
  AWQ_GEMV_CASE(8, 128)
  AWQ_GEMV_CASE(8, 64)
  AWQ_GEMV_CASE(8, 32)
#undef AWQ_GEMV_CASE
  set_error("awq_gemv: w_bit = %d, group = %d is not supported", w_bit, group);
  return AWQ_ERR_UNSUPPORTED;
}

}  // namespace awq
