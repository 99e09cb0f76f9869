// W4A16 decode matmul (M <= 8 tokens) for the default format: 4-bit codes in
// 128-channel groups with zero points.
//
// "awq-quantization（AWQ量化技术）Skill" page, section 主要功能和特点: a GEMV kernel
// serves batch-1 token generation; "AWQ量化实战" §3.4: decoding is bound by the
// bandwidth of reading the weights.
//
//  * Weights first.  A CTA owns a balanced range of output rows (and, when
//    the activations of the whole K do not fit in shared memory, a K slice of
//    a thread-block cluster).  Its warps (8 or 16) split the range's stages of 16
//    rows x 512 input channels (4 KB of codes as two 2 KB TMA boxes with the
//    128-byte swizzle, plus the stage's steps and zero points by 4-byte
//    cp.async) into contiguous runs, each warp streaming its run through its
//    own ring of slots, so that a warp only ever waits on its own slots, in
//    order.  Packed weights, steps and zero points never depend on the
//    previous kernel in the stream, so each warp fills its ring BEFORE
//    griddepcontrol.wait (programmatic dependent launch).  At one token two
//    8-warp CTAs of a launch share an SM.
//  * Dot products on the warp-level tensor-core MMA (mma.sync m16n8k16, fp16
//    operands, fp32 accumulation): the 16 weight rows of a stage are the A
//    operand, the (up to 8) tokens the N side.  On CUDA cores the same
//    reduction costs 8 FMA instructions per packed word; one MMA instruction
//    per word of each thread replaces them.  (A tcgen05 MMA costs ~57 issue
//    cycles per 128 x 16 x 16 instruction at N <= 16 whatever the width,
//    which caps it below the HBM rate of a decode step; this contraction is
//    HBM-bound, not flop-bound.)
//  * Dequantization: a lane's A fragment of one MMA holds four codes of row
//    g and four of row g + 8.  Lane (g, c) reads 16 contiguous bytes (32
//    channels) of each of its two rows per group, and one word feeds two
//    MMAs.  Codes become fp16 with one LOP3 per pair (1024 + q for the even
//    nibbles, 64 + q for the odd), HSUB2 of (1024 + z) or (64 + z) gives the
//    exact integer q - z.  Products x~ (q - z) are exact in fp32; each group's
//    sum is scaled by its step in fp32.  The activations are the B operand in
//    the matching order: a permutation of k applied to both operands leaves
//    every dot product unchanged.
//  * The scaled activations x~ = fp16(fp32(x) * inv_s) are built once per CTA
//    in shared memory, after the wait (they are the previous kernel's output).
//  * Results: a tile whose stages all fall in one warp's run is final in that
//    warp; a tile split between neighbouring warps is added in warp order
//    after one barrier, and K slices in cluster-rank order through
//    distributed shared memory.  The result is deterministic.
//  * Row ranges are not multiples of 16: a CTA's last tile is moved back to
//    end at the range's end, re-reading (from L2) rows the previous tile
//    already covered and discarding their results, so that no CTA reads rows
//    of another range.
#include <cooperative_groups.h>

#include "awq_internal.h"

namespace cg = cooperative_groups;

namespace awq {

__device__ unsigned int g_gemv_error = 0;
// Test hook (awq_debug_stall): the limit of every bounded wait, and a request
// that the first CTA withhold the TMA of its first stage, so that the wait
// for that stage runs out.
__device__ unsigned long long g_gemv_wait_ns = 1000000000ull;
__device__ unsigned int g_gemv_withhold = 0;

namespace {

constexpr int kStageK = 512;                      // input channels per stage
constexpr int kBoxBytes = 16 * 128;               // 16 rows x 32 words
constexpr int kStageBytes = 2 * kBoxBytes;        // codes of one stage
constexpr int kSideBytes = 16 * 8 + 16 * 4;       // steps [16][4] fp16, zero words [16]
constexpr int kMaxDepth = 8;
// Shared memory of one CTA when two CTAs share an SM (228 KB per SM, 1 KB
// reserved per CTA), and when one CTA has the SM.
constexpr int kHalfSmBytes = (228 * 1024) / 2 - 1024;
constexpr int kFullSmBytes = 227 * 1024;

__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(magic));
  return d;
}

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// d = A * B + c, m16n8k16, fp16 A (row) and B (col), fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A * B (fresh accumulators, no C operand registers to clear).
__device__ __forceinline__ void mma16816_first(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// Bounded wait on a phase of `bar`; the limit is read only once the first
// test has failed (the hot path keeps no register for it).  False when the
// limit ran out.
__device__ __forceinline__ bool wait_stage(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_bounded(bar, parity, *const_cast<volatile unsigned long long*>(&g_gemv_wait_ns));
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

// Arrives on `bar` once every cp.async issued so far by this thread has landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}


// Layout of a CTA's dynamic shared memory (byte offsets from a 1024-aligned
// base).  Computed identically on the host (size) and the device (offsets).
struct MmaLayout {
  int codes, side, bars, xs, part, tot, bytes;
  __host__ __device__ MmaLayout(int warps, int depth, int M, int KS, int rows_cap) {
    codes = 0;                                            // [warps][depth][4096]
    side = codes + warps * depth * kStageBytes;           // [warps][depth][192]
    bars = side + warps * depth * kSideBytes;             // [warps][depth] u64
    xs = ((bars + warps * depth * 8) + 15) & ~15;         // [M][KS * 2 + 64] bytes
    part = xs + M * (KS * 2 + 64);                        // [warps][2][M][16] fp32
    tot = part + warps * 2 * M * 16 * 4;                  // [rows_cap][M] fp32
    bytes = tot + rows_cap * M * 4 + 1024;                // + alignment slack
  }
};

// kWarps warps, each streaming its own contiguous run of stages through its
// own ring (a warp waits only on its own slots, in order); MINB CTAs per SM
// for the register budget; kDepth slots per ring (0: the run-time depth_rt),
// a constant for the plans the library uses so that the slot and phase
// arithmetic of every stage folds away.
template <int kWarps, int MINB, int kDepth>
__global__ void __launch_bounds__(kWarps * 32, MINB)
    gemv_mma_kernel(const __grid_constant__ CUtensorMap tq, const __half* __restrict__ X,
                    const __half* __restrict__ scales, const uint32_t* __restrict__ zeros,
                    const float* __restrict__ inv_s, int M, int N, int K, int KS, int depth_rt,
                    int rows_cap, __half* __restrict__ Y) {
  constexpr int kThreads = kWarps * 32;
  const int depth = kDepth > 0 ? kDepth : depth_rt;
  extern __shared__ uint8_t smem_raw[];
  // the 128-byte swizzle of the TMA boxes follows shared-memory address bits
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const MmaLayout L(kWarps, depth, M, KS, rows_cap);
  uint8_t* codes = smem + L.codes;
  uint8_t* side = smem + L.side;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint8_t* xsb = smem + L.xs;
  float* part = reinterpret_cast<float*>(smem + L.part);
  float* tot = reinterpret_cast<float*>(smem + L.tot);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  // MMA row g reads tile row pg (and g + 8 reads pg + 8): rows pg of the
  // lanes 0-7 of a shared-memory phase (g = 2p, 2p + 1) are p and p + 4,
  // whose swizzled 16-byte chunks fall in opposite halves of the banks.
  const int pg = ((g & 1) << 2) | (g >> 1);

  const int G = K / 128, ZW = (G + 7) / 8;
  const int r0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * N / gridDim.x);
  const int r1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * N / gridDim.x);
  const int nrows = r1 - r0;
  const int T = (nrows + 15) / 16;                       // row tiles
  const int kbeg = blockIdx.y * KS;
  const int klen = min(K - kbeg, KS);
  const int C = (klen + kStageK - 1) / kStageK;          // stages per tile
  const int S = T * C;
  const int sb = warp * S / kWarps, se = (warp + 1) * S / kWarps;   // S * kWarps < 2^31
  const int xstride = (KS / 128) * 256 + 64;             // bytes per token row of x~

  // first physical row of tile t: the last tile ends at r1 (may start below r0)
  auto tile_start = [&](int t) { return min(r0 + 16 * t, r1 - 16); };

  uint8_t* my_codes = codes + warp * depth * kStageBytes;
  uint8_t* my_side = side + warp * depth * kSideBytes;
  uint64_t* my_bars = bars + warp * depth;

  // Issue cursor: the next stage of the run to load, as (tile, chunk, slot),
  // with this lane's step and zero-point sources for the tile (row lane / 2
  // for the steps of groups 2 (lane % 2) .. + 1, row lane for the zero
  // points); a row below 0 (a tile reaching below the first row) loads none.
  int it = sb / C, ij = sb - (sb / C) * C, islot = 0, next = sb, its = 0;
  const __half* s_src = nullptr;
  const uint32_t* z_src = nullptr;
  auto set_tile = [&]() {
    its = tile_start(it);
    const int ps = its + (lane >> 1), pz = its + lane;
    s_src = ps >= 0 ? scales + static_cast<size_t>(ps) * G + (lane & 1) * 2 : nullptr;
    z_src = (lane < 16 && pz >= 0) ? zeros + static_cast<size_t>(pz) * ZW : nullptr;
  };
  set_tile();
  // Issues the stage at the cursor into its slot and advances the cursor;
  // withhold (the test hook only): the stage's codes are never requested.
  auto issue = [&](bool withhold) {
    const int kc = kbeg + ij * kStageK;
    const bool full = kbeg + klen - kc >= kStageK;       // 4 groups, else 2
    uint8_t* cb = my_codes + islot * kStageBytes;
    uint8_t* sd = my_side + islot * kSideBytes;
    uint64_t* bar = my_bars + islot;
    if (!withhold && elect_one()) {
      mbar_arrive_expect_tx(bar, full ? 2 * kBoxBytes : kBoxBytes);
      tma_load_2d(cb, &tq, bar, kc >> 3, its);
      if (full) tma_load_2d(cb + kBoxBytes, &tq, bar, (kc >> 3) + 32, its);
    }
    const int grp0 = kc >> 7;
    if (s_src && (full || !(lane & 1))) cp_async4(sd + lane * 4, s_src + grp0);
    if (z_src) cp_async4(sd + 128 + lane * 4, z_src + (grp0 >> 3));
    cp_async_arrive(bar);
    ++next;
    if (++islot == depth) islot = 0;
    if (++ij == C) {
      ij = 0;
      ++it;
      set_tile();
    }
  };

  // ---- before the dependency wait: barriers, then the first stages of the
  // warp's ring (weights only)
  if (lane == 0) {
    for (int s2 = 0; s2 < depth; ++s2) mbar_init(my_bars + s2, 33);
    fence_mbar_init();
    if (warp == 0) prefetch_tmap(&tq);
  }
  __syncwarp();
  {
    // the warp whose run holds the first stage of the first CTA
    bool withhold = g_gemv_withhold != 0 && blockIdx.x == 0 && blockIdx.y == 0 && sb == 0 &&
                    se > 0;
    while (next < se && next < sb + depth) {
      issue(withhold);
      withhold = false;
    }
  }

  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The next grid is released at once: its CTAs can only start where one of
  // this launch's CTAs has left (the launch's CTAs fill the register file),
  // so they take each SM the moment it frees without waiting for the launch
  // itself (measured: 0.6% faster on the 7B decode step than releasing it
  // after this CTA's last load).
  asm volatile("griddepcontrol.launch_dependents;");

  // ---- x~ = fp16(fp32(x) * inv_s) of the K slice.  Token m's row starts at
  // m * xstride bytes (odd tokens 64 bytes off the 128-byte grid, so the two
  // tokens a shared-memory phase reads use opposite bank halves); vector v
  // (8 channels k = 128 gl + 32 cc + 8 jj + i) sits at gl * 256 + jj * 64 +
  // cc * 16 and holds the pairs (k0,k4) (k1,k5) (k2,k6) (k3,k7) that the
  // dequantization produces
  const int nv = klen / 8;
  // x~ of token m, 8-channel vector v (inv_s given as is[], 1 when absent)
  auto put = [&](int m, int v, const uint4& xr, const float (&is)[8]) {
    const __half2* xh = reinterpret_cast<const __half2*>(&xr);
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t2 = __half22float2(xh[i]);
      f[2 * i] = __fmul_rn(t2.x, is[2 * i]);
      f[2 * i + 1] = __fmul_rn(t2.y, is[2 * i + 1]);
    }
    uint4 o;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 p2 = __halves2half2(__float2half_rn(f[i]), __float2half_rn(f[i + 4]));
      ow[i] = *reinterpret_cast<const uint32_t*>(&p2);
    }
    const int gl = v >> 4, cc = (v >> 2) & 3, jj = v & 3;
    *reinterpret_cast<uint4*>(xsb + m * xstride + gl * 256 + jj * 64 + cc * 16) = o;
  };
  auto load_is = [&](int k, float (&is)[8]) {
    if (inv_s) {
      const float4 ia = __ldg(reinterpret_cast<const float4*>(inv_s + k));
      const float4 ib = __ldg(reinterpret_cast<const float4*>(inv_s + k + 4));
      is[0] = ia.x; is[1] = ia.y; is[2] = ia.z; is[3] = ia.w;
      is[4] = ib.x; is[5] = ib.y; is[6] = ib.z; is[7] = ib.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) is[i] = 1.f;
    }
  };
  if (M <= 2) {
    // Up to kBatch (token, vector) items per thread have their loads in
    // flight together (the loads wait behind the weight stream in L2: one
    // latency per batch)
    const int nitems = M * nv;
    constexpr int kBatch = 4;
    for (int base = threadIdx.x; base < nitems; base += kThreads * kBatch) {
      uint4 xr[kBatch];
      float is[kBatch][8];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int q = base + u * kThreads;
        if (q < nitems) {
          const int m = q / nv, v = q - m * nv;
          const int k = kbeg + 8 * v;
          xr[u] = __ldg(reinterpret_cast<const uint4*>(X + static_cast<size_t>(m) * K + k));
          load_is(k, is[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int q = base + u * kThreads;
        if (q >= nitems) break;
        const int m = q / nv;
        put(m, q - m * nv, xr[u], is[u]);
      }
    }
  } else {
    // one vector of every token per thread and round: inv_s read once per
    // vector, all M loads in flight together
    for (int v = threadIdx.x; v < nv; v += kThreads) {
      const int k = kbeg + 8 * v;
      float is[8];
      load_is(k, is);
      uint4 xr[8];
#pragma unroll
      for (int m = 0; m < 8; ++m)
        if (m < M) xr[m] = __ldg(reinterpret_cast<const uint4*>(X + static_cast<size_t>(m) * K + k));
#pragma unroll
      for (int m = 0; m < 8; ++m)
        if (m < M) put(m, v, xr[m], is);
    }
  }
  __syncthreads();

  // token whose activations this lane supplies to the B operand: g when it
  // exists; otherwise any token of g's parity (its column is discarded)
  const int tg = g < M ? g : (M == 1 ? 0 : (g & 1));
  const uint8_t* xlane = xsb + tg * xstride + c * 16;
  // this lane's 16-byte chunk of rows pg and pg + 8 in a box, for the even
  // and the odd group of the box (128-byte swizzle: chunk ^ (row % 8))
  const int qoff0 = pg * 128 + ((c ^ pg) << 4);
  const int qoff1 = pg * 128 + (((4 | c) ^ pg) << 4);

  // first tile of this warp's run; a tile wholly inside the run is final here
  const int tf = sb / C;
  int failed_at = -1;   // stage whose wait ran out
  float acc[4] = {0.f, 0.f, 0.f, 0.f};

  auto flush = [&](int t) {
    const int ts = tile_start(t);
    const int own0 = r0 + 16 * t;
    const bool whole = t * C >= sb && (t + 1) * C <= se;
    const int slot = t == tf ? 0 : 1;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int row = pg + ((e >> 1) << 3);              // tile row
      const int tok = 2 * c + (e & 1);
      if (tok >= M) continue;
      if (whole) {
        if (ts + row >= own0) tot[(ts + row - r0) * M + tok] = acc[e];
      } else {
        part[((warp * 2 + slot) * M + tok) * 16 + row] = acc[e];
      }
    }
  };

  // consume cursor: stage i of the run is (tile ct, chunk cj) in slot cslot
  int ct = tf, cj = sb - tf * C, cslot = 0;
  uint32_t cphase = 0;
  for (int i = sb; i < se; ++i) {
    if (!wait_stage(my_bars + cslot, cphase)) {
      if (lane == 0) atomicOr(&g_gemv_error, 1u);
      failed_at = i;
      break;
    }
    const uint8_t* cb = my_codes + cslot * kStageBytes;
    const uint8_t* sd = my_side + cslot * kSideBytes;
    const int kc = kbeg + cj * kStageK;
    float s_a[4], s_b[4];   // steps of the stage's groups, rows pg and pg + 8
    {
      const uint2 ua = *reinterpret_cast<const uint2*>(sd + pg * 8);
      const uint2 ub = *reinterpret_cast<const uint2*>(sd + (pg + 8) * 8);
      const float2 a01 = __half22float2(*reinterpret_cast<const __half2*>(&ua.x));
      const float2 a23 = __half22float2(*reinterpret_cast<const __half2*>(&ua.y));
      const float2 b01 = __half22float2(*reinterpret_cast<const __half2*>(&ub.x));
      const float2 b23 = __half22float2(*reinterpret_cast<const __half2*>(&ub.y));
      s_a[0] = a01.x; s_a[1] = a01.y; s_a[2] = a23.x; s_a[3] = a23.y;
      s_b[0] = b01.x; s_b[1] = b01.y; s_b[2] = b23.x; s_b[3] = b23.y;
    }
    const int zsh = (kc >> 5) & 16;                       // group kc / 128 mod 8 is 0 or 4
    const uint32_t za_w = *reinterpret_cast<const uint32_t*>(sd + 128 + pg * 4) >> zsh;
    const uint32_t zb_w = *reinterpret_cast<const uint32_t*>(sd + 128 + (pg + 8) * 4) >> zsh;
    const uint8_t* xst = xlane + ((kc - kbeg) << 1);      // 256 bytes per group
    // one group h of the stage: 8 MMAs over 16 rows x 128 channels
    auto group = [&](int h) {
      const uint8_t* qp = cb + (h >> 1) * kBoxBytes + ((h & 1) ? qoff1 : qoff0);
      const uint4 qa = *reinterpret_cast<const uint4*>(qp);
      const uint4 qb = *reinterpret_cast<const uint4*>(qp + 8 * 128);
      const uint32_t za = (za_w >> (4 * h)) & 15u, zb = (zb_w >> (4 * h)) & 15u;
      const uint32_t zae = za * 0x00010001u + 0x64006400u, zao = za * 0x00100010u + 0x54005400u;
      const uint32_t zbe = zb * 0x00010001u + 0x64006400u, zbo = zb * 0x00100010u + 0x54005400u;
      const uint8_t* xg = xst + h * 256;
      float d0[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const uint32_t wa = jj == 0 ? qa.x : jj == 1 ? qa.y : jj == 2 ? qa.z : qa.w;
        const uint32_t wb = jj == 0 ? qb.x : jj == 1 ? qb.y : jj == 2 ? qb.z : qb.w;
        const uint4 xv = *reinterpret_cast<const uint4*>(xg + jj * 64);
        const uint32_t ta = wa >> 8, tb = wb >> 8;
        const uint32_t a0 = hsub2_u(and_or(wa, 0x000F000Fu, 0x64006400u), zae);   // (k0,k4)
        const uint32_t a1 = hsub2_u(and_or(wa, 0x00F000F0u, 0x54005400u), zao);   // (k1,k5)
        const uint32_t a2 = hsub2_u(and_or(ta, 0x000F000Fu, 0x64006400u), zae);   // (k2,k6)
        const uint32_t a3 = hsub2_u(and_or(ta, 0x00F000F0u, 0x54005400u), zao);   // (k3,k7)
        const uint32_t b0 = hsub2_u(and_or(wb, 0x000F000Fu, 0x64006400u), zbe);
        const uint32_t b1 = hsub2_u(and_or(wb, 0x00F000F0u, 0x54005400u), zbo);
        const uint32_t b2 = hsub2_u(and_or(tb, 0x000F000Fu, 0x64006400u), zbe);
        const uint32_t b3 = hsub2_u(and_or(tb, 0x00F000F0u, 0x54005400u), zbo);
        // logical k (2c, 2c+1) <- (k0, k4), (2c+8, 2c+9) <- (k1, k5); and (k2, k6), (k3, k7)
        if (jj == 0) mma16816_first(d0, a0, b0, a1, b1, xv.x, xv.y);
        else mma16816(d0, a0, b0, a1, b1, xv.x, xv.y);
        mma16816(d0, a2, b2, a3, b3, xv.z, xv.w);
      }
      acc[0] = fmaf(s_a[h], d0[0], acc[0]);
      acc[1] = fmaf(s_a[h], d0[1], acc[1]);
      acc[2] = fmaf(s_b[h], d0[2], acc[2]);
      acc[3] = fmaf(s_b[h], d0[3], acc[3]);
    };
    if (kbeg + klen - kc >= kStageK) {
#pragma unroll
      for (int h = 0; h < 4; ++h) group(h);
    } else {   // the last stage of a slice ending 256 channels into it
#pragma unroll
      for (int h = 0; h < 2; ++h) group(h);
    }
    __syncwarp();
    if (next < se) {
      fence_proxy_async_smem();
      issue(false);
    }
    if (++cslot == depth) {
      cslot = 0;
      cphase ^= 1u;
    }
    if (++cj == C) {   // the tile is done
      flush(ct);
      cj = 0;
      ++ct;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] = 0.f;
    }
  }
  if (failed_at >= 0) {
    // drain the copies still in flight into this warp's ring (bounded): the
    // stages failed_at .. next - 1 are in the slots from cslot on
    for (int i = failed_at; i < next; ++i) {
      wait_stage(my_bars + cslot, cphase);
      if (++cslot == depth) {
        cslot = 0;
        cphase ^= 1u;
      }
    }
  } else if (cj > 0 && se > sb) {
    flush(ct);   // the run ends inside tile ct
  }
  __syncthreads();

  // ---- tiles split between warps: add the partial sums in warp order
  for (int idx = threadIdx.x; idx < T * M * 16; idx += kThreads) {
    const int t = idx / (M * 16), rem = idx - t * M * 16;
    const int tok = rem >> 4, row = rem & 15;
    const int ts = tile_start(t);
    if (ts + row < r0 + 16 * t) continue;                // not owned by this tile
    const int s0 = t * C, s1 = (t + 1) * C;              // stages of the tile
    float v = 0.f;
    int nw = 0;
    bool whole = false;
    for (int w = 0; w < kWarps; ++w) {
      const int wb = w * S / kWarps, we = (w + 1) * S / kWarps;   // S * kWarps < 2^31
      if (we <= s0 || wb >= s1 || wb == we) continue;
      if (wb <= s0 && we >= s1) {
        whole = true;
        break;
      }
      const int slot = (wb / C) == t ? 0 : 1;
      v += part[((w * 2 + slot) * M + tok) * 16 + row];
      ++nw;
    }
    if (!whole && nw > 0) tot[(ts + row - r0) * M + tok] = v;
  }
  __syncthreads();

  if (gridDim.y == 1) {
    for (int i = threadIdx.x; i < M * nrows; i += kThreads) {
      const int m = i / nrows, r = i - m * nrows;
      Y[static_cast<size_t>(m) * N + r0 + r] = __float2half_rn(tot[r * M + m]);
    }
    return;
  }
  // ---- K split over the cluster: rank 0 adds the CTA totals in rank order
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  if (cluster.block_rank() == 0) {
    for (int i = threadIdx.x; i < M * nrows; i += kThreads) {
      const int m = i / nrows, r = i - m * nrows;
      float v = 0.f;
      for (int rk = 0; rk < static_cast<int>(gridDim.y); ++rk)
        v += cluster.map_shared_rank(tot, rk)[r * M + m];
      Y[static_cast<size_t>(m) * N + r0 + r] = __float2half_rn(v);
    }
  }
  cluster.sync();   // every CTA's shared memory stays alive until rank 0 has read it
}

}  // namespace

// A plan with `warps` warps and `ctas_per_sm` CTAs of one launch per SM
// (grid = SMs x ctas_per_sm over the rows): the smallest K split whose
// activations leave room for rings of at least `min_depth` stages per warp,
// with the deepest ring (up to max_depth) that fits.  depth 0 when none fits.
MmaGemvPlan make_gemv_mma_plan(int M, int N, int K, int sms, int warps, int ctas_per_sm,
                               int min_depth, int max_depth) {
  MmaGemvPlan p{};
  const int budget = ctas_per_sm == 2 ? kHalfSmBytes : kFullSmBytes;
  if (max_depth > kMaxDepth) max_depth = kMaxDepth;
  for (int nsplit = 1; nsplit <= 8; nsplit *= 2) {
    const int nst = (K / kStageK + ((K % kStageK) ? 1 : 0));   // stages along K
    const int per = (nst + nsplit - 1) / nsplit;
    const int KS = per * kStageK;
    const int ns = (K + KS - 1) / KS;
    int gx = sms * ctas_per_sm / ns;
    const int tiles = (N + 15) / 16;
    if (gx > tiles) gx = tiles;
    if (gx < 1) gx = 1;
    const int rows_cap = (N + gx - 1) / gx;
    for (int depth = max_depth; depth >= min_depth; --depth) {
      const MmaLayout L(warps, depth, M, KS, rows_cap);
      if (L.bytes <= budget) {
        p.warps = warps;
        p.depth = depth;
        p.nsplit = ns;
        p.KS = KS;
        p.gx = gx;
        p.rows_cap = rows_cap;
        p.smem = L.bytes;
        p.ctas_per_sm = ctas_per_sm;
        return p;
      }
    }
  }
  return p;
}

// The launch plan the library uses, in order of preference (measured on the
// Llama-2 decode shapes): two CTAs of eight warps per SM, each warp with a
// ring of two 4 KB stages (fastest at M = 1, against deeper rings, one CTA of
// 8, 12 or 16 warps per SM, and one CTA beside the next launch's); when the
// activations of several tokens do not fit half an SM, one CTA of sixteen
// warps per SM (the activations once per SM), with K halved over a cluster of
// two and then with 1-deep rings if needed (70B qkv and 7B down at 8 tokens);
// wider K splits over a cluster only when none of these fits.
MmaGemvPlan plan_gemv_mma(int M, int N, int K, int sms) {
  MmaGemvPlan p = make_gemv_mma_plan(M, N, K, sms, 8, 2, 2, 2);
  if (p.depth > 0 && p.nsplit == 1) return p;
  // one 16-warp CTA per SM: the whole K, else K halved over a cluster of two,
  // with 2-deep rings, else with 1-deep ones (16 stages in flight per SM)
  const MmaGemvPlan q = make_gemv_mma_plan(M, N, K, sms, 16, 1, 2, 2);
  if (q.depth > 0 && q.nsplit <= 2) return q;
  const MmaGemvPlan q1 = make_gemv_mma_plan(M, N, K, sms, 16, 1, 1, 1);
  if (q1.depth > 0 && q1.nsplit <= 2) return q1;
  if (p.depth == 0) p = make_gemv_mma_plan(M, N, K, sms, 8, 1, 2, kMaxDepth);
  return p;
}

bool gemv_mma_eligible(int M, int K, int w_bit, int group, bool silu_mul) {
  return !silu_mul && w_bit == 4 && group == 128 && M >= 1 && M <= 8 && K % 256 == 0;
}

namespace {
template <int W, int MINB, int D>
int launch_mma(const MmaGemvPlan& p, const CUtensorMap& tq, const __half* X, int M,
               const __half* scales, const uint32_t* zeros, const float* inv_s, int N, int K,
               __half* Y, cudaStream_t st) {
  auto kern = gemv_mma_kernel<W, MINB, D>;
  const int rc = ensure_smem_attr(reinterpret_cast<const void*>(kern), p.smem);
  if (rc != AWQ_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.gx, p.nsplit, 1);
  cfg.blockDim = dim3(W * 32, 1, 1);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = p.nsplit;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.nsplit > 1 ? 2 : 1;
  AWQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, tq, X, scales, zeros, inv_s, M, N, K, p.KS,
                                  p.depth, p.rows_cap, Y));
  return AWQ_OK;
}
}  // namespace

int launch_gemv_mma_plan(const MmaGemvPlan& p, const __half* X, int M, const uint32_t* qweight,
                         const __half* scales, const uint32_t* zeros, const float* inv_s, int N,
                         int K, __half* Y, cudaStream_t st) {
  if (p.depth == 0) {
    set_error("awq_gemv: no shared-memory plan for M = %d, N = %d, K = %d", M, N, K);
    return AWQ_ERR_SHAPE;
  }
  CUtensorMap tq;
  const int rc = make_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT32, qweight,
                              static_cast<uint64_t>(K) / 8, static_cast<uint64_t>(N),
                              static_cast<uint64_t>(K) / 2, 32, 16, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != AWQ_OK) return rc;
#define AWQ_MMA_CASE(W, B, D)                                                                  \
  if (p.warps == W && p.ctas_per_sm == B && (D == 0 || p.depth == D))                          \
    return launch_mma<W, B, D>(p, tq, X, M, scales, zeros, inv_s, N, K, Y, st);
  AWQ_MMA_CASE(8, 2, 2)
  AWQ_MMA_CASE(16, 1, 2)
  AWQ_MMA_CASE(16, 1, 1)
  AWQ_MMA_CASE(8, 2, 0)
  AWQ_MMA_CASE(8, 1, 0)
  AWQ_MMA_CASE(16, 1, 0)
#undef AWQ_MMA_CASE
  set_error("awq_gemv: no kernel for %d warps at %d CTAs per SM", p.warps, p.ctas_per_sm);
  return AWQ_ERR_UNSUPPORTED;
}

int launch_gemv_mma(const __half* X, int M, const uint32_t* qweight, const __half* scales,
                    const uint32_t* zeros, const float* inv_s, int N, int K, __half* Y,
                    cudaStream_t st) {
  return launch_gemv_mma_plan(plan_gemv_mma(M, N, K, sm_count()), X, M, qweight, scales, zeros,
                              inv_s, N, K, Y, st);
}

int set_gemv_stall(int withhold, uint64_t wait_ns) {
  const unsigned w = withhold ? 1u : 0u;
  const unsigned long long ns = wait_ns;
  AWQ_CUDA_TRY(cudaMemcpyToSymbol(g_gemv_withhold, &w, sizeof(w)));
  AWQ_CUDA_TRY(cudaMemcpyToSymbol(g_gemv_wait_ns, &ns, sizeof(ns)));
  return AWQ_OK;
}

int read_clear_gemv_error(cudaStream_t st, unsigned* flags) {
  AWQ_CUDA_TRY(cudaStreamSynchronize(st));
  unsigned v = 0, zero = 0;
  AWQ_CUDA_TRY(cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(v)));
  AWQ_CUDA_TRY(cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(zero)));
  *flags = v;
  return AWQ_OK;
}

}  // namespace awq
