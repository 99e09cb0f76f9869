// W4A16 matmul for few tokens (M <= 128) on the 5th-generation tensor cores.
//
// "awq-quantization（AWQ量化技术）Skill" page, section 主要功能和特点: the GEMM
// kernel serves batch > 1.  With a handful of tokens the layer reads every
// packed weight once and does little arithmetic with it, so the launch is
// bound by how fast 128 x K weight tiles can be fetched and turned into MMA
// operands, not by the tensor cores.  This kernel is built for that:
//
//  * a stage covers 128 input channels (64 for 8-bit codes or 64-channel
//    groups), so every fixed cost of a stage (barriers, fences, copies
//    issued) is paid per 8 KB of packed codes;
//  * the dequantized weight operand lives in tensor memory, not shared
//    memory: the MMA takes A from tensor memory (row i of the tile in lane
//    i), which removes the 4x-expanded fp16 tile's write and read from the
//    shared-memory bandwidth; shared memory only holds the packed codes and
//    the activation tile, in a deep ring (16..24 stages) released by the MMA;
//  * three teams (two at 64 and 128 tokens) of four dequantization warps
//    take the stages in turn, each thread one whole weight row of its stage
//    (16 or 8 chunks of 8 codes), written with tcgen05.st into a ring of
//    4..8 operand stages;
//  * the operand holds the exact integers q - z (HSUB2 of fp16 magic
//    numbers, no rounding), and each group's partial product accumulates in
//    its own tensor-memory accumulator (a ring of four, two at 128 tokens);
//    the epilogue warps read it, multiply by the group's step s in fp32 and
//    add it to the output row they keep in registers.  That takes the
//    multiply by s off the per-weight path and leaves only the final fp32
//    sum to round.
//
// A 128 x BN x 16 MMA costs about as much for BN = 16 as for BN = 64 (a
// fixed ~57 cycles plus ~0.4 cycle per token column, measured on B300), so
// the tensor pipe bounds this kernel at about 8 x 60 cycles per 8 KB stage.
//
//   y[m][n] = sum_g s[n][g] * sum_{k in g} (q[n][k] - z[n][g]) * x~[m][k]
//
// Warp roles: warp 0 issues TMA (codes [128 rows x 16 words], activations
// [BN x 64] per 64 channels, 128-byte swizzle); warp 1 allocates tensor
// memory and issues tcgen05.mma (one thread); the next 12 (8) warps
// dequantize; the last 4 (8 at 128 tokens) run the per-group epilogue.
// Every mbarrier wait is bounded (1 s); on expiry the kernel records the fact
// in a device word, makes the other roles stop, drains its copies and MMAs,
// frees tensor memory and returns.
#include "awq_internal.h"

namespace awq {

__device__ unsigned int g_narrow_error = 0;

namespace {

constexpr int NBM = 128;                  // weight rows per tile (MMA M)
constexpr uint64_t kNWaitNs = 1000000000ull;
constexpr int kNSmemBudget = 227 * 1024;

template <int BN, int BITS, int BKS>
struct NCfg {
  // dequantization teams of 4 warps: three while the epilogue's output row
  // (BN registers) is short, two at BN = 64 to stay clear of spills
  static constexpr int TEAMS = BN <= 32 ? 3 : 2;
  static constexpr int DEQ_WARPS = 4 * TEAMS;
  // epilogue: 4 warps (one per tensor-memory lane quarter), 8 at BN = 128,
  // each pair of a quarter taking half of the token columns
  static constexpr int EPI_WARPS = BN == 128 ? 8 : 4;
  static constexpr int EPI_COLS = BN * 4 / EPI_WARPS;
  static constexpr int THREADS = 32 * (2 + DEQ_WARPS + EPI_WARPS);
  static constexpr int NATOM = BKS / 64;                // 128-byte swizzle atoms per row
  static constexpr int RAW_ROW = BKS * BITS / 8;        // packed bytes of a row per stage
  static constexpr int RAW_BYTES = NBM * RAW_ROW;
  static constexpr int B_BYTES = BN * BKS * 2;
  static constexpr int RSLOT = RAW_BYTES + B_BYTES;     // codes + activation tile
  static constexpr int CTRL = 1024;                     // barriers, tmem slot, flag
  static constexpr int SR_FIT = (kNSmemBudget - 1024 - CTRL) / RSLOT;
  static constexpr int SR = SR_FIT > 24 ? 24 : SR_FIT;
  // tensor memory (512 columns): NRING group accumulators (groups in flight
  // between the MMA and the epilogue), then the operand ring, BKS / 2
  // columns (two fp16 per column) per stage
  static constexpr int ACC_COLS = BN < 32 ? 32 : BN;
  static constexpr int NRING = BN == 128 ? 2 : 4;
  static constexpr int A_COL0 = NRING * ACC_COLS;
  static constexpr int A_COLS = BKS / 2;
  static constexpr int SA_FIT = (512 - A_COL0) / A_COLS;
  static constexpr int SA = SA_FIT > 8 ? 8 : SA_FIT;
  static constexpr int TMEM_COLS = 512;
  static constexpr int SMEM = 1024 + SR * RSLOT + CTRL;
  static_assert(SR >= 4 && SA >= 3, "ring depths");
  static_assert(SMEM <= kNSmemBudget, "shared memory");
  static_assert(RAW_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "1024-byte aligned tiles");
};

struct NAbort {
  volatile int* flag;
  __device__ bool raised() const { return *flag != 0; }
  __device__ void raise(unsigned bit) const {
    *flag = 1;
    atomicOr(&g_narrow_error, bit);
  }
};

__device__ __forceinline__ bool nwait(uint64_t* bar, uint32_t parity, const NAbort& ab,
                                      unsigned bit) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (ab.raised()) return false;
    if (globaltimer_ns() - t0 > kNWaitNs) {
      ab.raise(bit);
      return false;
    }
  }
}

// 8 4-bit codes of one word -> 8 fp16 integers q - z.  Magic fp16 numbers:
// 1024 + q for the even nibbles of each 16-bit half and 64 + q for the odd
// ones; HSUB2 of (1024 + z) or (64 + z) gives q - z exactly.  With PERM the
// 16 output bytes hold the pairs (k0,k4) (k1,k5) (k2,k6) (k3,k7), the chunk
// order of the prescaled activations; otherwise k is natural.
template <bool PERM>
__device__ __forceinline__ uint4 codes4_minus_zero(uint32_t w, uint32_t zbe, uint32_t zbo) {
  const uint32_t t = w >> 8;
  const uint32_t h0 = (w & 0x000F000Fu) | 0x64006400u;   // (k0, k4)
  const uint32_t h1 = (w & 0x00F000F0u) | 0x54005400u;   // (k1, k5)
  const uint32_t h2 = (t & 0x000F000Fu) | 0x64006400u;   // (k2, k6)
  const uint32_t h3 = (t & 0x00F000F0u) | 0x54005400u;   // (k3, k7)
  uint32_t p[4], zz[4];
  if (PERM) {
    p[0] = h0; p[1] = h1; p[2] = h2; p[3] = h3;
    zz[0] = zbe; zz[1] = zbo; zz[2] = zbe; zz[3] = zbo;
  } else {
    p[0] = __byte_perm(h0, h1, 0x5410);   // (k0, k1)
    p[1] = __byte_perm(h2, h3, 0x5410);   // (k2, k3)
    p[2] = __byte_perm(h0, h1, 0x7632);   // (k4, k5)
    p[3] = __byte_perm(h2, h3, 0x7632);   // (k6, k7)
    const uint32_t zmix = __byte_perm(zbe, zbo, 0x5410);
    zz[0] = zmix; zz[1] = zmix; zz[2] = zmix; zz[3] = zmix;
  }
  uint4 out;
  uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 d = __hsub2(*reinterpret_cast<const __half2*>(&p[i]),
                              *reinterpret_cast<const __half2*>(&zz[i]));
    o[i] = *reinterpret_cast<const uint32_t*>(&d);
  }
  return out;
}

// Two words of 8-bit codes (k0..k7) -> 8 fp16 integers q - z (magic 1024 + q
// for both bytes of each 16-bit half after one shift).  With PERM the pairs
// are (k0,k2) (k1,k3) (k4,k6) (k5,k7); otherwise k is natural.
template <bool PERM>
__device__ __forceinline__ uint4 codes8_minus_zero(uint32_t w0, uint32_t w1, uint32_t zb) {
  uint32_t p[4];
  p[0] = (w0 & 0x00FF00FFu) | 0x64006400u;          // (k0, k2)
  p[1] = ((w0 >> 8) & 0x00FF00FFu) | 0x64006400u;   // (k1, k3)
  p[2] = (w1 & 0x00FF00FFu) | 0x64006400u;          // (k4, k6)
  p[3] = ((w1 >> 8) & 0x00FF00FFu) | 0x64006400u;   // (k5, k7)
  if (!PERM) {
    const uint32_t a = p[0], b = p[1], c = p[2], d = p[3];
    p[0] = __byte_perm(a, b, 0x5410);
    p[1] = __byte_perm(a, b, 0x7632);
    p[2] = __byte_perm(c, d, 0x5410);
    p[3] = __byte_perm(c, d, 0x7632);
  }
  uint4 out;
  uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 d = __hsub2(*reinterpret_cast<const __half2*>(&p[i]),
                              *reinterpret_cast<const __half2*>(&zb));
    o[i] = *reinterpret_cast<const uint32_t*>(&d);
  }
  return out;
}

// One launch: work item t covers tile t / splits (128 output channels n0..
// x BN tokens m0..) over the stages [kb0, kb1) of split t % splits (kps
// stages of BKS channels each, a whole number of groups).  gs_shift =
// log2(group), spg_shift = log2(group / BKS).
template <int BN, bool PERM, int BITS, int BKS>
__global__ void __launch_bounds__(NCfg<BN, BITS, BKS>::THREADS, 1)
    gemm_narrow_kernel(const __grid_constant__ CUtensorMap tm_x,
                       const __grid_constant__ CUtensorMap tm_q,
                       const __half* __restrict__ scales, const uint32_t* __restrict__ zeros,
                       int M, int N, int K, int gs_shift, int spg_shift,
                       __half* __restrict__ out, int ldo, int splits, int kps,
                       float* __restrict__ part) {
  using C = NCfg<BN, BITS, BKS>;
  constexpr int SR = C::SR;
  constexpr int SA = C::SA;
  constexpr int PW = 32 / BITS;                  // codes per packed word
  constexpr int PW_SHIFT = BITS == 4 ? 3 : 2;
  constexpr uint32_t QMASK = (1u << BITS) - 1u;
  constexpr int KWS = BKS * BITS / 32;           // packed words of a row per stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sR = smem;                                  // [SR][codes | activations]
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(sR + SR * C::RSLOT);
  uint64_t* raw_empty = raw_full + SR;
  uint64_t* a_full = raw_empty + SR;
  uint64_t* a_empty = a_full + SA;
  uint64_t* g_full = a_empty + SA;
  uint64_t* g_empty = g_full + C::NRING;
  uint64_t* drain = g_empty + C::NRING;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const NAbort ab{abort_flag};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = K / BKS;
  const int n_tiles = (N + NBM - 1) / NBM;
  const int items = n_tiles * ((M + BN - 1) / BN) * splits;
  const int spg_mask = (1 << spg_shift) - 1;
  auto krange = [&](int t, int& kb0, int& kb1) {
    kb0 = (t % splits) * kps;
    kb1 = kb0 + kps < nk ? kb0 + kps : nk;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < SR; ++s) {
      mbar_init(raw_full + s, 1);
      mbar_init(raw_empty + s, 1);
    }
    for (int s = 0; s < SA; ++s) {
      mbar_init(a_full + s, 4);                     // one arrival per warp of a team
      mbar_init(a_empty + s, 1);
    }
    for (int b = 0; b < C::NRING; ++b) {
      mbar_init(g_full + b, 1);
      mbar_init(g_empty + b, 32 * C::EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_q);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // programmatic stream serialization: every global read comes after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // the whole warp walks the stages; one elected lane issues the copies
    int it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < items && ok; t += gridDim.x) {
      const int tile = t / splits;
      const int n0 = (tile % n_tiles) * NBM, m0 = (tile / n_tiles) * BN;
      int kb0, kb1;
      krange(t, kb0, kb1);
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int s = it % SR;
        const bool got = it < SR || nwait(raw_empty + s, ((it / SR) - 1) & 1, ab, 1u);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        uint8_t* slot = sR + s * C::RSLOT;
        if (elect_one()) {
          mbar_arrive_expect_tx(raw_full + s, C::RSLOT);
          tma_load_2d(slot, &tm_q, raw_full + s, kb * KWS, n0);
#pragma unroll
          for (int a = 0; a < C::NATOM; ++a)
            tma_load_2d(slot + C::RAW_BYTES + a * (BN * 128), &tm_x, raw_full + s,
                        kb * BKS + a * 64, m0);
        }
        __syncwarp();
      }
    }
    // copies still in flight complete before the CTA may exit
    for (int j = it > SR ? it - SR : 0; j < it; ++j) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(raw_full + j % SR, (j / SR) & 1))
        if (globaltimer_ns() - t0 > kNWaitNs) {
          ab.raise(16u);
          break;
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp walks the stages; one elected lane issues the MMAs.
    // Any shared-memory access of this warp, an mbarrier wait included,
    // waits until the MMAs it has queued drain (~160 cycles, measured), so
    // it waits on one barrier per stage: a_full, which the dequantization
    // team arrives on only after it has seen the stage's codes and
    // activations land (raw_full) and, at a group's first stage, the
    // group's accumulator freed by the epilogue (g_empty).
    constexpr uint32_t idesc = idesc_f16_f32(NBM, BN);
    int it = 0, gcount = 0, slot = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < items && ok; t += gridDim.x) {
      int kb0, kb1;
      krange(t, kb0, kb1);
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int rs = it % SR, as = it % SA;
        const bool first = (kb & spg_mask) == 0;
        if (first) slot = gcount % C::NRING;
        const bool got = nwait(a_full + as, (it / SA) & 1, ab, 2u);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_tmem = tmem + C::A_COL0 + as * C::A_COLS;
        const uint64_t bd = sw128_kmajor_desc(smem_u32(sR + rs * C::RSLOT + C::RAW_BYTES));
        const uint32_t d_tmem = tmem + slot * C::ACC_COLS;
        const bool last = ((kb + 1) & spg_mask) == 0;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BKS / 16; ++kk)
            umma_f16_ts(d_tmem, a_tmem + kk * 8, bd + (kk >> 2) * (BN * 128 >> 4) + 2 * (kk & 3),
                        idesc, (first && kk == 0) ? 0u : 1u);
          umma_commit(a_empty + as);
          umma_commit(raw_empty + rs);
          if (last) umma_commit(g_full + slot);
        }
        __syncwarp();
        if (last) ++gcount;
      }
    }
    if (elect_one()) umma_commit(drain);
    __syncwarp();
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(drain, 0))
      if (globaltimer_ns() - t0 > kNWaitNs) {
        ab.raise(32u);
        break;
      }
    __syncwarp();
  } else if (warp < 2 + C::DEQ_WARPS) {
    // ------------------------------------------------------------ dequant
    const int dw = warp - 2;
    const int team = dw >> 2;
    // a warp reaches tensor-memory lanes 32 (warp % 4) .. + 31: row r = lane r
    const int r = (warp & 3) * 32 + lane;
    const int G = K >> gs_shift, ZW = (G + PW - 1) / PW;
    constexpr int NQ = C::RAW_ROW / 16;            // 16-byte pieces of a row's codes
    // the code tile arrives with the TMA's 64-byte (32-byte) swizzle: piece p
    // of row r sits at p ^ ((r >> 1) & 3) (p ^ ((r >> 2) & 1)), so the 8
    // threads of a shared-memory wavefront read 8 different bank groups
    const int swz = (r / (128 / C::RAW_ROW)) % NQ;
    int it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < items && ok; t += gridDim.x) {
      const int n = ((t / splits) % n_tiles) * NBM + r;
      const bool row_ok = n < N;
      const uint32_t* zrow = zeros + static_cast<size_t>(row_ok ? n : 0) * ZW;
      auto zload = [&](int w) -> uint32_t { return (row_ok && w < ZW) ? __ldg(zrow + w) : 0u; };
      int kb0, kb1;
      krange(t, kb0, kb1);
      const int it0 = it;
      // this team's first stage of the item: (it0 + kb - kb0) % TEAMS == team
      constexpr int kTeams = C::TEAMS;
      int kb = kb0 + ((team - it0) % kTeams + kTeams) % kTeams;
      int zwi = ((kb * BKS) >> gs_shift) >> PW_SHIFT;
      uint32_t zcur = zload(zwi), znext = zload(zwi + 1);
      for (; kb < kb1; kb += kTeams) {
        const int sit = it0 + (kb - kb0);
        const int g = (kb * BKS) >> gs_shift;
        const int wi = g >> PW_SHIFT;
        if (wi != zwi) {
          zcur = wi == zwi + 1 ? znext : zload(wi);
          znext = zload(wi + 1);
          zwi = wi;
        }
        const uint32_t zc = (zcur >> ((g & (PW - 1)) * BITS)) & QMASK;
        const uint32_t zbe = (0x6400u | zc) * 0x00010001u;          // (1024 + z) x 2
        const uint32_t zbo = (0x5400u | (zc << 4)) * 0x00010001u;   // (64 + z) x 2, 4-bit
        const int rs = sit % SR, as = sit % SA;
        bool got = nwait(raw_full + rs, (sit / SR) & 1, ab, 4u);
        if (got && sit >= SA) got = nwait(a_empty + as, ((sit / SA) - 1) & 1, ab, 4u);
        // the first stage of a group also waits until the epilogue has freed
        // the group's accumulator, so that the MMA warp waits on a_full alone
        // (groups never straddle items, so the CTA's group ordinal is
        // sit >> spg_shift)
        const int gidx = sit >> spg_shift;
        if (got && (kb & spg_mask) == 0 && gidx >= C::NRING)
          got = nwait(g_empty + gidx % C::NRING, ((gidx / C::NRING) - 1) & 1, ab, 4u);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* rp = sR + rs * C::RSLOT + r * C::RAW_ROW;
        const uint32_t a_tmem =
            tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + C::A_COL0 + as * C::A_COLS;
        // each 16-byte piece gives 4 (4-bit) or 2 (8-bit) chunks of 8
        // channels, 4 tensor-memory columns per chunk
#pragma unroll
        for (int p = 0; p < NQ; ++p) {
          const uint4 v = *reinterpret_cast<const uint4*>(rp + ((p ^ swz) << 4));
          uint32_t cols[BITS == 4 ? 16 : 8];
          if constexpr (BITS == 4) {
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 o = codes4_minus_zero<PERM>(wv[i], zbe, zbo);
              cols[4 * i] = o.x; cols[4 * i + 1] = o.y; cols[4 * i + 2] = o.z; cols[4 * i + 3] = o.w;
            }
            tmem_st16(a_tmem + p * 16, cols);
          } else {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const uint4 o = codes8_minus_zero<PERM>(i ? v.z : v.x, i ? v.w : v.y, zbe);
              cols[4 * i] = o.x; cols[4 * i + 1] = o.y; cols[4 * i + 2] = o.z; cols[4 * i + 3] = o.w;
            }
            tmem_st8(a_tmem + p * 8, cols);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(a_full + as);
      }
      it = it0 + (kb1 - kb0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;                  // tensor-memory lanes 32q .. 32q + 31
    constexpr int EC = C::EPI_COLS;
    const int cb = ((warp - 2 - C::DEQ_WARPS) >> 2) * EC;   // first token column
    const int G = K >> gs_shift;
    int gcount = 0;
    for (int t = blockIdx.x; t < items; t += gridDim.x) {
      const int tile = t / splits;
      const int n0 = (tile % n_tiles) * NBM, m0 = (tile / n_tiles) * BN;
      const int n = n0 + quarter * 32 + lane;
      const bool row_ok = n < N;
      const __half* srow = scales + static_cast<size_t>(row_ok ? n : 0) * G;
      int kb0, kb1;
      krange(t, kb0, kb1);
      const int g0 = (kb0 * BKS) >> gs_shift, g1 = (kb1 * BKS) >> gs_shift;
      constexpr int AHEAD = 4;
      float sq[AHEAD];
#pragma unroll
      for (int i = 0; i < AHEAD; ++i)
        sq[i] = (row_ok && g0 + i < g1) ? __half2float(srow[g0 + i]) : 0.f;
      float y[EC];
#pragma unroll
      for (int j = 0; j < EC; ++j) y[j] = 0.f;
      bool ok = true;
      for (int g = g0; g < g1; ++g, ++gcount) {
        const int slot = gcount % C::NRING;
        const bool got = nwait(g_full + slot, (gcount / C::NRING) & 1, ab, 8u);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float s = sq[0];
#pragma unroll
        for (int i = 0; i + 1 < AHEAD; ++i) sq[i] = sq[i + 1];
        sq[AHEAD - 1] = (row_ok && g + AHEAD < g1) ? __half2float(srow[g + AHEAD]) : 0.f;
        const uint32_t gaddr =
            tmem + slot * C::ACC_COLS + cb + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll
        for (int c0 = 0; c0 < EC; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(gaddr + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) y[c0 + j] = fmaf(s, __uint_as_float(v[j]), y[c0 + j]);
        }
        tc_fence_before();
        mbar_arrive(g_empty + slot);
      }
      if (!ok) break;
      float* pout = part + static_cast<size_t>(t % splits) * M * ldo;   // splits > 1
#pragma unroll
      for (int j = 0; j < EC; ++j) {
        const int m = m0 + cb + j;
        if (m < M && row_ok) {
          const size_t idx = static_cast<size_t>(m) * ldo + n;
          if (splits > 1)
            pout[idx] = y[j];
          else
            out[idx] = __float2half_rn(y[j]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int BN, bool PERM, int BITS, int BKS>
int launch_narrow_tile(const CUtensorMap& tx, const CUtensorMap& tq, const __half* scales,
                       const uint32_t* zeros, int M, int N, int K, int gs_shift, int spg_shift,
                       __half* out, int ldo, int splits, int kps, float* part,
                       cudaStream_t st) {
  using C = NCfg<BN, BITS, BKS>;
  {
    const int rc = ensure_smem_attr(
        reinterpret_cast<const void*>(gemm_narrow_kernel<BN, PERM, BITS, BKS>), C::SMEM);
    if (rc != AWQ_OK) return rc;
  }
  const int sms = sm_count();
  const int items = ((N + NBM - 1) / NBM) * ((M + BN - 1) / BN) * splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(items < sms ? items : sms, 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  AWQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, gemm_narrow_kernel<BN, PERM, BITS, BKS>, tx, tq, scales,
                                  zeros, M, N, K, gs_shift, spg_shift, out, ldo, splits, kps,
                                  part));
  if (splits > 1) return launch_splitk_reduce(part, splits, M, N, out, st);
  return AWQ_OK;
}

template <bool PERM, int BITS, int BKS>
int dispatch_narrow(int bn, const CUtensorMap& tx, const CUtensorMap& tq, const __half* scales,
                    const uint32_t* zeros, int M, int N, int K, int gs_shift, int spg_shift,
                    __half* out, int ldo, int splits, int kps, float* part, cudaStream_t st) {
  switch (bn) {
    case 16:
      return launch_narrow_tile<16, PERM, BITS, BKS>(tx, tq, scales, zeros, M, N, K, gs_shift,
                                                     spg_shift, out, ldo, splits, kps, part, st);
    case 32:
      return launch_narrow_tile<32, PERM, BITS, BKS>(tx, tq, scales, zeros, M, N, K, gs_shift,
                                                     spg_shift, out, ldo, splits, kps, part, st);
    case 64:
      return launch_narrow_tile<64, PERM, BITS, BKS>(tx, tq, scales, zeros, M, N, K, gs_shift,
                                                     spg_shift, out, ldo, splits, kps, part, st);
    default:
      return launch_narrow_tile<128, PERM, BITS, BKS>(tx, tq, scales, zeros, M, N, K, gs_shift,
                                                      spg_shift, out, ldo, splits, kps, part, st);
  }
}

int stage_channels(int w_bit, int group) { return (w_bit == 4 && group == 128) ? 128 : 64; }

}  // namespace

bool narrow_eligible(int M, int w_bit, int group) {
  return M >= 1 && M <= kNarrowMaxM && (w_bit == 4 || w_bit == 8) &&
         (group == 128 || group == 64);
}

// Token tile and split-K, from a cost model in SM cycles fitted to B300
// measurements (the 7B and 70B layer shapes at 8..64 tokens, splits 1..8):
// a stage of a work item costs ~1000 (1 + M / 500) cycles per 8 KB of packed
// codes (the rate one SM sustains; far from the HBM bound, so it is the
// number of stages the busiest SM walks that counts); items run in rounds of
// one per SM; a split-K plan pays ~4000 cycles for the second launch and
// 16 bytes per output per split of fp32 partial sums at ~3250 bytes per
// cycle.  Splits come in whole groups, 1, 2, 3, 4, 6 or 8 of them.
NarrowPlan plan_narrow(int M, int N, int K, int w_bit, int group) {
  NarrowPlan p{0, 1, 0, 0};
  if (!narrow_eligible(M, w_bit, group)) return p;
  const int bks = stage_channels(w_bit, group);
  const int spg = group / bks;
  const int nk = K / bks;
  const int bn = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
  const int sms = sm_count();
  const int tiles = ((N + NBM - 1) / NBM) * ((M + bn - 1) / bn);
  const double stage_cycles =
      1000.0 * (1.0 + M / 500.0) * (128.0 * bks * w_bit / 8.0) / 8192.0;
  double best_t = -1.0;
  for (const int s : {1, 2, 3, 4, 6, 8}) {
    int kps = (nk + s - 1) / s;
    kps = (kps + spg - 1) / spg * spg;
    if (s > 1 && kps < 4 * spg) break;
    if ((nk + kps - 1) / kps != s) continue;
    const int rounds = (tiles * s + sms - 1) / sms;
    double t = static_cast<double>(rounds) * kps * stage_cycles;
    if (s > 1) t += 4000.0 + 16.0 * s * static_cast<double>(M) * N / 3250.0;
    if (best_t < 0 || t < best_t) {
      best_t = t;
      p = NarrowPlan{bn, s, kps, bks};
    }
  }
  return p;
}

size_t narrow_partial_bytes(int M, int N, int K) {
  size_t most = 0;
  const int cfgs[3][2] = {{4, 128}, {4, 64}, {8, 128}};   // the three stage/group shapes
  for (const auto& c : cfgs) {
    const NarrowPlan p = plan_narrow(M, N, K, c[0], c[1]);
    if (p.bn && p.splits > 1) {
      const size_t b = static_cast<size_t>(p.splits) * M * N * sizeof(float);
      if (b > most) most = b;
    }
  }
  return most;
}

int launch_gemm_narrow(const __half* Xt, bool xt_permuted, int M, const uint32_t* qweight,
                       const __half* scales, const uint32_t* zeros, int N, int K, __half* out,
                       int ldo, cudaStream_t st, int w_bit, int group, float* part,
                       size_t part_bytes) {
  NarrowPlan plan = plan_narrow(M, N, K, w_bit, group);
  if (!plan.bn) {
    set_error("awq_gemm: no narrow-token plan for M = %d, w_bit = %d, group = %d", M, w_bit,
              group);
    return AWQ_ERR_UNSUPPORTED;
  }
  if (plan.splits > 1 &&
      (!part || part_bytes < static_cast<size_t>(plan.splits) * M * N * sizeof(float) ||
       ldo != N || !aligned16(part))) {
    plan.splits = 1;
    plan.kps = K / plan.bks;
  }
  const int bks = plan.bks;
  CUtensorMap tx, tq;
  int rc = make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Xt, K, M,
                        static_cast<uint64_t>(K) * 2, 64, plan.bn, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != AWQ_OK) return rc;
  const int pw = 32 / w_bit;
  const int raw_row = bks * w_bit / 8;   // 64 or 32 bytes
  rc = make_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT32, qweight, K / pw, N,
                    static_cast<uint64_t>(K / pw) * 4, raw_row / 4, NBM,
                    raw_row == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  if (rc != AWQ_OK) return rc;
  const int gs_shift = group == 128 ? 7 : 6;
  const int spg_shift = group / bks == 2 ? 1 : 0;
  if (w_bit == 8) {
    if (xt_permuted)
      return dispatch_narrow<true, 8, 64>(plan.bn, tx, tq, scales, zeros, M, N, K, gs_shift,
                                          spg_shift, out, ldo, plan.splits, plan.kps, part, st);
    return dispatch_narrow<false, 8, 64>(plan.bn, tx, tq, scales, zeros, M, N, K, gs_shift,
                                         spg_shift, out, ldo, plan.splits, plan.kps, part, st);
  }
  if (bks == 128) {
    if (xt_permuted)
      return dispatch_narrow<true, 4, 128>(plan.bn, tx, tq, scales, zeros, M, N, K, gs_shift,
                                           spg_shift, out, ldo, plan.splits, plan.kps, part, st);
    return dispatch_narrow<false, 4, 128>(plan.bn, tx, tq, scales, zeros, M, N, K, gs_shift,
                                          spg_shift, out, ldo, plan.splits, plan.kps, part, st);
  }
  if (xt_permuted)
    return dispatch_narrow<true, 4, 64>(plan.bn, tx, tq, scales, zeros, M, N, K, gs_shift,
                                        spg_shift, out, ldo, plan.splits, plan.kps, part, st);
  return dispatch_narrow<false, 4, 64>(plan.bn, tx, tq, scales, zeros, M, N, K, gs_shift,
                                       spg_shift, out, ldo, plan.splits, plan.kps, part, st);
}

int read_clear_narrow_error(cudaStream_t st, unsigned* flags) {
  AWQ_CUDA_TRY(cudaStreamSynchronize(st));
  unsigned v = 0, zero = 0;
  AWQ_CUDA_TRY(cudaMemcpyFromSymbol(&v, g_narrow_error, sizeof(v)));
  AWQ_CUDA_TRY(cudaMemcpyToSymbol(g_narrow_error, &zero, sizeof(zero)));
  *flags = v;
  return AWQ_OK;
}

}  // namespace awq
