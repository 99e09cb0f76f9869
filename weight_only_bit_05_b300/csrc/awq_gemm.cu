// W4A16 matmul on the 5th-generation tensor cores (tcgen05), any M.
//
// "awq-quantization（AWQ量化技术）Skill" page, section 主要功能和特点: the GEMM kernel
// serves batch > 1 and prefill.  There the layer is a dense contraction, so
// it runs on the tensor cores:
//
//   D[n][m] = sum_k W^'[n][k] * X~[m][k]       (MMA M = 128 weight rows,
//                                               MMA N = BN tokens, K = 16/step)
//
// The kernel is persistent: one CTA per SM walks the (128 output channels x
// BN tokens) tiles of Y^T with warp roles.  Above 128 tokens (BN = 160) the
// dequantized operand lives in tensor memory:
//   warp 0       TMA producer (warp-converged, one elected lane): packed codes
//                [128 rows x 16 words] and the activation tile as two [160 x
//                64] boxes (128-byte swizzle) per 128-channel stage, into a
//                4-stage ring, completion counted on full[s];
//   warp 1       allocates tensor memory (two 160-column accumulators and three
//                64-column operand stages) and issues tcgen05.mma with A from
//                tensor memory, 8 per stage (warp-converged, one elected
//                lane), releasing the stage through tcgen05.commit -> empty[s],
//                the operand stage -> a_empty[a] and a finished accumulator
//                -> acc_full[b];
//   warps 2..25  three teams of 8 taking stages in turn: each thread turns 32
//                channels of one row per k-block into w^ = (q - z) * s (half2)
//                and writes them into its warp's lane quarter of the team's
//                operand stage (tcgen05.st), then arrives on a_full[a];
//   warps 26-29  epilogue: read a finished accumulator from tensor memory
//                (tcgen05.ld), write the outputs and free it (acc_empty[b]),
//                while the next tile accumulates into the other buffer.
// At BN <= 128 and for the squared-error and dense passes of the scale
// search (BN = 256) the operand goes through shared memory instead: 64-channel
// stages, 8 dequantization warps writing the 128-byte-swizzled K-major layout
// (deq[s]), both MMA operands read from shared memory, 4 epilogue warps.
// Putting the weights on the MMA's M side means every CTA dequantizes its
// 128 x K weight tile exactly once per BN tokens, and small token counts
// (BN = 16) waste no tensor-core work on padding.  Consecutive tiles of the
// walk share the activation tile, which stays in L2.
//
// Every wait on an mbarrier is bounded (1 s); a wait that runs out records
// the fact in a device word (read by awq_check_device_error), makes the
// other roles stop, drains the copies and MMAs in flight, frees tensor
// memory and returns.
#include "awq_internal.h"

namespace awq {

__device__ unsigned int g_gemm_error = 0;
// Test hook (awq_debug_stall): the limit of every bounded wait, and a request
// that the producer of the first CTA withhold the copies of its first stage.
__device__ unsigned long long g_gemm_wait_ns = 1000000000ull;
__device__ unsigned int g_gemm_withhold = 0;

namespace {

constexpr int BM = 128;          // weight rows per CTA (MMA M)
constexpr int BK = 64;           // K per stage: one 128-byte swizzle atom of fp16
constexpr int kEpiWarps = 4;
// limit of the bounded waits, read only on their slow path
__device__ __forceinline__ uint64_t wait_limit_ns() {
  return *const_cast<volatile unsigned long long*>(&g_gemm_wait_ns);
}
constexpr int kSmemBudget = 227 * 1024 - 2048;

// At BN = 160 the dequantized operand does not pass through shared memory:
// the dequantization warps write it into a ring in tensor memory (after the
// two 160-column accumulators) and the MMA reads A from there.  Shared memory
// then carries only the activation tile and the packed codes of a stage.
// Measured on B300, neither shared memory nor L2 bounds either layout (bank
// and crossbar counters stay below 40%); what bounds them is the chain of
// copy, dequantization and MMA issue within a CTA, and the tensor-memory
// operand shortens that chain (the MMA issues from a converged warp in ~46
// cycles with A in tensor memory, ~70 with A in shared memory) and lets
// several dequantization teams fill separate operand stages.
template <int BN, int MODE, int BITS>
struct Cfg {
  static constexpr bool ATM = BN == 160;
  // 64-channel k-blocks per pipeline stage: two with A in tensor memory, so
  // that every wait, commit and arrive of the roles serves 8 MMAs, not 4
  static constexpr int SK = ATM ? 2 : 1;
  static constexpr int A_BYTES = ATM ? 0 : BM * BK * 2;
  static constexpr int B_SUB = BN * BK * 2;         // one 64-channel column of activations
  static constexpr int B_BYTES = B_SUB * SK;
  static constexpr int RAW_ROW = BK * SK * BITS / 8;   // packed bytes of one row per stage
  static constexpr int RAW_BYTES = (MODE == kGemmDenseF32) ? 0 : BM * RAW_ROW;
  static constexpr int STAGE = A_BYTES + B_BYTES + RAW_BYTES;
  static constexpr int STAGES = (kSmemBudget / STAGE) > 8 ? 8 : (kSmemBudget / STAGE);
  static constexpr int ACC_COLS = BN < 32 ? 32 : BN;   // one fp32 accumulator
  // double-buffered accumulators (the epilogue of a tile overlaps the next
  // tile's MMAs); with A in tensor memory the A ring follows them:
  // 2 x 160 + 3 stages x 64 columns
  static constexpr int ACC_BUFS = 2;
  static constexpr int TMEM_COLS = ATM ? 512 : 2 * ACC_COLS;
  static constexpr int A_COL0 = ACC_BUFS * ACC_COLS;      // A ring (ATM): first column
  static constexpr int A_COLS = BK * SK / 2;              // columns of one stage of A
  static constexpr int A_STAGES = ATM ? (512 - A_COL0) / A_COLS : 1;
  // dequantization warps: 8 cover a k-block (4 lane quarters x 2 halves of
  // its 64 channels); with A in tensor memory three such teams take the
  // stages in turn, each into its own stage of the A ring, so that two teams
  // dequantize while the MMA consumes the third team's stage (a team's
  // dequantization of a stage takes longer than the stage's MMAs)
  static constexpr int DEQ_TEAMS = ATM ? 3 : 1;
  static_assert(!ATM || A_STAGES == DEQ_TEAMS, "A ring: one stage per dequantization team");
  static constexpr int DEQ_WARPS = 8 * DEQ_TEAMS;
  static constexpr int THREADS = 64 + 32 * (DEQ_WARPS + kEpiWarps);
  static constexpr int SMEM = STAGES * STAGE + 1024 + 512;
};

struct Abort {
  volatile int* flag;
  __device__ bool raised() const { return *flag != 0; }
  __device__ void raise(unsigned bit) const {
    *flag = 1;
    atomicOr(&g_gemm_error, bit);
  }
};

// Bounded wait that also gives up as soon as another role has aborted.  The
// waiting thread sleeps in the barrier (suspend hint) rather than polling:
// the tensor-memory lane quarter of a warp is also its scheduler, so each
// scheduler runs two dequantization warps beside an epilogue warp and (on two
// of them) the producer or the MMA thread, and a polling waiter would take
// issue slots from the dequantization it is waiting for.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const Abort& ab,
                                              unsigned bit) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (ab.raised()) return false;
    if (globaltimer_ns() - t0 > wait_limit_ns()) {
      ab.raise(bit);
      return false;
    }
  }
}

// 8 codes of one word -> 8 fp16 weights (q - z) * s.  Magic fp16 numbers:
// 1024 + q for the even nibbles (bits 0..3 of each 16-bit half) and 64 + q for
// the odd ones (bits 4..7), so a single shift serves all four pairs; HSUB2 of
// the matching (1024 + z) or (64 + z) gives q - z exactly and HMUL2 rounds the
// product to fp16 once.  With PERM the 16 output bytes hold the pairs (k0,k4)
// (k1,k5) (k2,k6) (k3,k7), the order in which the prescale kernel lays out
// each 8-element chunk of the activations (a permutation of k applied to both
// MMA operands leaves every dot product unchanged); otherwise k is natural.
template <bool PERM>
__device__ __forceinline__ uint4 dequant_word(uint32_t w, uint32_t zbe, uint32_t zbo,
                                              __half2 s2) {
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
                              *reinterpret_cast<const __half2*>(&zz[i]));   // q - z, exact
    const __half2 v = __hmul2(d, s2);
    o[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return out;
}

// Two 8-bit words (codes k0..k7) -> 8 fp16 weights (q - z) * s: bytes 0 and 2
// of a word (bits 0..7 of each 16-bit half) and, after one shift, bytes 1 and
// 3 become the fp16 number 1024 + q; HSUB2 and HMUL2 as for 4-bit codes.
// With PERM the output pairs are (k0,k2) (k1,k3) (k4,k6) (k5,k7), the order of
// the prescale kernel's 8-bit chunk layout; otherwise k is natural.
template <bool PERM>
__device__ __forceinline__ uint4 dequant_word8(uint32_t w0, uint32_t w1, uint32_t zb, __half2 s2) {
  uint32_t p[4];
  p[0] = (w0 & 0x00FF00FFu) | 0x64006400u;          // (k0, k2)
  p[1] = ((w0 >> 8) & 0x00FF00FFu) | 0x64006400u;   // (k1, k3)
  p[2] = (w1 & 0x00FF00FFu) | 0x64006400u;          // (k4, k6)
  p[3] = ((w1 >> 8) & 0x00FF00FFu) | 0x64006400u;   // (k5, k7)
  if (!PERM) {
    const uint32_t a = p[0], b = p[1], c = p[2], d = p[3];
    p[0] = __byte_perm(a, b, 0x5410);   // (k0, k1)
    p[1] = __byte_perm(a, b, 0x7632);   // (k2, k3)
    p[2] = __byte_perm(c, d, 0x5410);   // (k4, k5)
    p[3] = __byte_perm(c, d, 0x7632);   // (k6, k7)
  }
  uint4 out;
  uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 dd = __hsub2(*reinterpret_cast<const __half2*>(&p[i]),
                               *reinterpret_cast<const __half2*>(&zb));   // q - z, exact
    const __half2 v = __hmul2(dd, s2);
    o[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return out;
}

// Steps and zero points run this many groups ahead of the dequantization, so
// that their global loads never wait on the memory latency.
constexpr int kSzAhead = 4;

template <int BN, int MODE, bool PERM, int BITS>
__global__ void __launch_bounds__(Cfg<BN, MODE, BITS>::THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_a,
                const __half* __restrict__ scales, const uint32_t* __restrict__ zeros, int M,
                int N, int K, int gs, void* __restrict__ out, int ldo,
                const float* __restrict__ yref, int ldy, int full_tiles, int ts, int kps,
                float* __restrict__ part) {
  using C = Cfg<BN, MODE, BITS>;
  constexpr int KWB = BK * BITS / 32;   // packed words of one row per stage
  constexpr int S = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * C::A_BYTES;
  uint8_t* sRaw = sB + S * C::B_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sRaw + S * C::RAW_BYTES);
  uint64_t* deq = full + S;
  uint64_t* empty = deq + S;
  uint64_t* acc_full = empty + S;     // [2]
  uint64_t* acc_empty = acc_full + 2; // [2]
  uint64_t* drain = acc_empty + 2;
  uint64_t* a_full = drain + 1;             // [A_STAGES] (ATM)
  uint64_t* a_empty = a_full + C::A_STAGES; // [A_STAGES] (ATM)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(a_empty + C::A_STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const Abort ab{abort_flag};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = K / BK;
  const int n_tiles = (N + BM - 1) / BM;
  const int tiles = n_tiles * ((M + BN - 1) / BN);
  // Work items: items t < full_tiles are the whole tiles 0 .. full_tiles - 1
  // (fp16 output); the remaining tiles are split over K, ts ways each: item
  // full_tiles + u is part u % ts of tile full_tiles + u / ts, k-blocks
  // [kb0, kb1), kps of them (an even number, so that no part starts inside
  // a 128-channel group; the host guarantees every part is non-empty).  A
  // part writes fp32 partial sums to its own [BN][BM] block of `part` and a
  // second kernel adds a tile's parts in order.  Plain split-K over every
  // tile is full_tiles = 0; no split at all is ts = 1.
  const int items = full_tiles + (tiles - full_tiles) * ts;
  auto item_of = [&](int t, int& tile, int& kb0, int& kb1, int& split) {
    if (t < full_tiles) {
      tile = t;
      split = -1;
      kb0 = 0;
      kb1 = nk;
      return;
    }
    const int u = t - full_tiles, q = u / ts;
    tile = full_tiles + q;
    split = ts > 1 ? u - q * ts : -1;
    kb0 = ts > 1 ? (u - q * ts) * kps : 0;
    kb1 = ts > 1 && kb0 + kps < nk ? kb0 + kps : nk;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, 1);
      mbar_init(deq + s, 32 * 8);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full + b, 1);
      mbar_init(acc_empty + b, 32 * kEpiWarps);
    }
    mbar_init(drain, 1);
    if (C::ATM)
      for (int a = 0; a < C::A_STAGES; ++a) {
        mbar_init(a_full + a, 32 * 8);
        mbar_init(a_empty + a, 1);
      }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // launched with programmatic stream serialization: the setup above may
  // overlap the previous kernel; every global read comes after this wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // (warp-converged like the MMA issuer; one elected lane issues the copies)
    {
      int it = 0;   // k-blocks issued by this CTA over all its tiles
      bool ok = true;
      // test hook: the first stage of the first CTA is never requested
      const bool withhold = g_gemm_withhold != 0 && blockIdx.x == 0;
      for (int t = blockIdx.x; t < items && ok; t += gridDim.x) {
        int tile, kb0, kb1, split;
        item_of(t, tile, kb0, kb1, split);
        const int n0 = (tile % n_tiles) * BM, m0 = (tile / n_tiles) * BN;
        for (int kb = kb0; kb < kb1; kb += C::SK, ++it) {
          const int s = it % S;
          if (it >= S &&
              !__all_sync(0xffffffffu, wait_or_abort(empty + s, ((it / S) - 1) & 1, ab, 1u))) {
            ok = false;
            break;
          }
          if (it == 0 && withhold) continue;
          if (elect_one()) {
            mbar_arrive_expect_tx(full + s, (MODE == kGemmDenseF32 ? C::A_BYTES : C::RAW_BYTES) +
                                                C::B_BYTES);
            if (MODE == kGemmDenseF32)
              tma_load_2d(sA + s * C::A_BYTES, &tm_a, full + s, kb * BK, n0);
            else if (MODE == kGemmSiluF16) {
              // 64 gate rows and the 64 matching up rows of the tile's pairs
              tma_load_2d(sRaw + s * C::RAW_BYTES, &tm_a, full + s, kb * KWB, n0 / 2);
              tma_load_2d(sRaw + s * C::RAW_BYTES + (BM / 2) * C::RAW_ROW, &tm_a, full + s,
                          kb * KWB, N / 2 + n0 / 2);
            } else {
              tma_load_2d(sRaw + s * C::RAW_BYTES, &tm_a, full + s, kb * KWB, n0);
            }
#pragma unroll
            for (int j = 0; j < C::SK; ++j)
              tma_load_2d(sB + s * C::B_BYTES + j * C::B_SUB, &tm_b, full + s, (kb + j) * BK, m0);
          }
          __syncwarp();
        }
      }
      // the copies still in flight complete before the CTA may exit
      for (int j = it > S ? it - S : 0; j < it; ++j) {
        const int s = j % S;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(full + s, (j / S) & 1))
          if (globaltimer_ns() - t0 > wait_limit_ns()) {
            if (lane == 0) ab.raise(16u);
            break;
          }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (its waits and descriptors warp-uniform)
    // and one elected lane issues: measured on B300, a tcgen05.mma issued
    // from a lone divergent thread costs about 96 cycles of issue, about 46
    // (A in tensor memory) to 70 from a converged warp, and a 128 x 160 x 16
    // MMA runs 80 cycles.  With A in tensor memory, a_full implies that the
    // stage's activations have landed (the dequantization warps saw `full`
    // before they arrived), so the MMA waits on a_full alone.
    {
      constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
      int it = 0, lt = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < items && ok; t += gridDim.x, ++lt) {
        const int b = lt % C::ACC_BUFS;
        if (lt >= C::ACC_BUFS &&
            !__all_sync(0xffffffffu, wait_or_abort(acc_empty + b, ((lt / C::ACC_BUFS) - 1) & 1,
                                                   ab, 2u)))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + b * C::ACC_COLS;
        int tile, kb0, kb1, split;
        item_of(t, tile, kb0, kb1, split);
        for (int kb = kb0; kb < kb1; kb += C::SK, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          const int as = it % C::A_STAGES;
          bool got;
          if constexpr (C::ATM) {
            got = wait_or_abort(a_full + as, (it / C::A_STAGES) & 1, ab, 2u);
          } else {
            got = wait_or_abort(full + s, ph, ab, 2u);
            if (got && MODE != kGemmDenseF32) got = wait_or_abort(deq + s, ph, ab, 2u);
          }
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd = sw128_kmajor_desc(smem_u32(sB + s * C::B_BYTES));
          if constexpr (C::ATM) {
            const uint32_t at = tmem + C::A_COL0 + as * C::A_COLS;
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < C::SK * BK / 16; ++kk)
                umma_f16_ts(d_tmem, at + kk * 8, bd + (kk >> 2) * (C::B_SUB >> 4) + 2 * (kk & 3),
                            idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
              umma_commit(empty + s);
              umma_commit(a_empty + as);
            }
          } else {
            const uint64_t ad = sw128_kmajor_desc(smem_u32(sA + s * C::A_BYTES));
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk)
                umma_f16(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc,
                         (kb != kb0 || kk != 0) ? 1u : 0u);
              umma_commit(empty + s);
            }
          }
          __syncwarp();
        }
        if (ok && elect_one()) umma_commit(acc_full + b);
        __syncwarp();
      }
      if (elect_one()) umma_commit(drain);
      __syncwarp();
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0))
        if (globaltimer_ns() - t0 > wait_limit_ns()) {
          if (lane == 0) ab.raise(32u);
          break;
        }
    }
    __syncwarp();
  } else if (warp < 2 + C::DEQ_WARPS) {
    // ------------------------------------------------------------ dequant
    if constexpr (C::ATM) {
      // Team `team` (8 warps) dequantizes the stages (two k-blocks each)
      // whose CTA-wide ordinal is `team` modulo the number of teams; a thread
      // covers 32 channels (`half`) of each k-block for one row of its warp's
      // tensor-memory lane quarter.
      const int d = warp - 2;                 // 0 .. DEQ_WARPS - 1
      const int team = d >> 3;
      const int half = (d >> 2) & 1;
      const int r = (warp & 3) * 32 + lane;   // tile row = tensor-memory lane
      constexpr int PW = 32 / BITS;           // codes per packed word
      constexpr uint32_t QMASK = (1u << BITS) - 1u;
      const int G = K / gs, ZW = (G + PW - 1) / PW;
      const int gshift = gs == 128 ? 7 : gs == 64 ? 6 : 5;
      // steps and zero points 8 groups at a time when rows hold whole blocks
      // of 8 groups, the block after the current one loaded ahead
      const bool blocks8 = (G % 8) == 0;
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < items && ok; t += gridDim.x) {
        int tile, kb0, kb1, split;
        item_of(t, tile, kb0, kb1, split);
        // with the fused gate/up weight, MMA row r of the tile is virtual row
        // v = n0 + r: gate row v/2 for even v, up row v/2 for odd v
        const int v = (tile % n_tiles) * BM + r;
        const int n = MODE == kGemmSiluF16 ? (v >> 1) + (v & 1) * (N / 2) : v;
        const bool row_ok = MODE == kGemmSiluF16 ? (v >> 1) < N / 2 : v < N;
        const int raw_r = MODE == kGemmSiluF16 ? (r >> 1) + (r & 1) * (BM / 2) : r;
        const __half* srow = scales + static_cast<size_t>(row_ok ? n : 0) * G;
        const uint32_t* zrow = zeros + static_cast<size_t>(row_ok ? n : 0) * ZW;
        uint4 sb0 = make_uint4(0, 0, 0, 0), sb1 = sb0;
        uint32_t z00 = 0, z01 = 0, z10 = 0, z11 = 0;
        auto load_blk = [&](int b, uint4& sb, uint32_t& za, uint32_t& zb) {
          if (row_ok && 8 * b < G) {
            sb = __ldg(reinterpret_cast<const uint4*>(srow + 8 * b));
            za = __ldg(zrow + (8 * b) / PW);
            zb = PW == 4 ? __ldg(zrow + (8 * b) / PW + 1) : 0u;
          } else {
            sb = make_uint4(0, 0, 0, 0);
            za = zb = 0u;
          }
        };
        int blk = -2, cur_g = -1;
        uint32_t zbe = 0x64006400u, zbo = 0x54005400u;
        __half2 s2 = __half2half2(__ushort_as_half(0));
        // step and zero point of group gi (groups only move forward)
        auto set_group = [&](int gi) {
          if (gi == cur_g) return;
          cur_g = gi;
          uint32_t zc;
          if (blocks8) {
            const int b = gi >> 3;
            if (b != blk) {
              if (b == blk + 1) {
                sb0 = sb1;
                z00 = z10;
                z01 = z11;
              } else {
                load_blk(b, sb0, z00, z01);
              }
              load_blk(b + 1, sb1, z10, z11);
              blk = b;
            }
            const int j = gi & 7;
            const uint32_t sw = (j >> 1) == 0 ? sb0.x : (j >> 1) == 1 ? sb0.y
                              : (j >> 1) == 2 ? sb0.z : sb0.w;
            s2 = __half2half2(__ushort_as_half(static_cast<unsigned short>(sw >> (16 * (j & 1)))));
            zc = PW == 8 ? (z00 >> (4 * j)) & QMASK
                         : (((j >> 2) == 0 ? z00 : z01) >> (8 * (j & 3))) & QMASK;
          } else {
            s2 = __half2half2(row_ok ? srow[gi] : __ushort_as_half(0));
            zc = row_ok ? (__ldg(zrow + gi / PW) >> ((gi % PW) * BITS)) & QMASK : 0u;
          }
          zbe = (0x6400u | zc) * 0x00010001u;          // (1024 + z, 1024 + z)
          zbo = (0x5400u | (zc << 4)) * 0x00010001u;   // (64 + z, 64 + z), 4-bit only
        };
        for (int kb = kb0; kb < kb1; kb += C::SK, ++it) {
          if (it % C::DEQ_TEAMS != team) continue;
          const int s = it % S;
          const int as = it % C::A_STAGES;
          // the warp stays converged for the tensor-memory stores
          bool got = wait_or_abort(full + s, (it / S) & 1, ab, 4u);
          if (got && it >= C::A_STAGES)
            got = wait_or_abort(a_empty + as, ((it / C::A_STAGES) - 1) & 1, ab, 4u);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ta = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + C::A_COL0 +
                              as * C::A_COLS + half * 16;
#pragma unroll
          for (int kl = 0; kl < C::SK; ++kl) {
            set_group(((kb + kl) * BK + half * 32) >> gshift);
            // this thread's 32 channels of k-block kb + kl
            const uint8_t* rp = sRaw + s * C::RAW_BYTES + raw_r * C::RAW_ROW +
                                kl * (C::RAW_ROW / C::SK) + half * (C::RAW_ROW / (2 * C::SK));
            uint32_t cols[16];
            if constexpr (BITS == 4) {
              const uint4 raw = *reinterpret_cast<const uint4*>(rp);
              const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint4 o = dequant_word<PERM>(rw[i], zbe, zbo, s2);
                cols[4 * i] = o.x; cols[4 * i + 1] = o.y; cols[4 * i + 2] = o.z; cols[4 * i + 3] = o.w;
              }
            } else {
              const uint4 r0 = *reinterpret_cast<const uint4*>(rp);
              const uint4 r1 = *reinterpret_cast<const uint4*>(rp + 16);
              const uint32_t rw[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint4 o = dequant_word8<PERM>(rw[2 * i], rw[2 * i + 1], zbe, s2);
                cols[4 * i] = o.x; cols[4 * i + 1] = o.y; cols[4 * i + 2] = o.z; cols[4 * i + 3] = o.w;
              }
            }
            tmem_st16(ta + kl * (BK / 2), cols);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(a_full + as);
        }
      }
    } else if (MODE != kGemmDenseF32) {
      const int d = warp - 2;                 // 0..7
      const int r = (warp & 3) * 32 + lane;   // tile row (= the warp's tensor-memory lanes)
      const int half = d >> 2;                // input channels 32*half .. +31 of the stage
      constexpr int PW = 32 / BITS;        // codes per packed word
      constexpr uint32_t QMASK = (1u << BITS) - 1u;
      const int G = K / gs, ZW = (G + PW - 1) / PW;
      // the groups this thread meets, in order: a new one every 2^kb_shift
      // stages (2 for 128-channel groups, else 1), gstride groups after the
      // previous one (2 for 32-channel groups, else 1); shifts, not divisions,
      // on this per-stage path
      const int kb_shift = gs > BK ? 1 : 0;
      const int kb_mask = (1 << kb_shift) - 1;
      const int gstride = gs >= BK ? 1 : BK / gs;
      const int gfirst = (half * 32) / gs;
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < items && ok; t += gridDim.x) {
        // with the fused gate/up weight, MMA row r of the tile is virtual row
        // v = n0 + r: gate row v/2 for even v, up row v/2 for odd v
        int tile, kb0, kb1, split;
        item_of(t, tile, kb0, kb1, split);
        const int v = (tile % n_tiles) * BM + r;
        const int n = MODE == kGemmSiluF16 ? (v >> 1) + (v & 1) * (N / 2) : v;
        const bool row_ok = MODE == kGemmSiluF16 ? (v >> 1) < N / 2 : v < N;
        const int raw_r = MODE == kGemmSiluF16 ? (r >> 1) + (r & 1) * (BM / 2) : r;
        // Steps and zero points.  When every row's groups come in whole
        // blocks of 8 (G % 8 == 0) and this thread meets every group, they
        // are read 8 at a time (one 16-byte load of steps, one or two words of
        // zero points) into two register blocks, the next block 8 groups ahead
        // of use; otherwise one group at a time, kSzAhead groups ahead.
        const bool blocks8 = (G % 8 == 0) && gstride == 1;
        uint4 sblk[2];
        uint32_t zblk[2][2];
        auto load_blk = [&](int b, int slot) {
          if (row_ok && 8 * b < G) {
            sblk[slot] = __ldg(reinterpret_cast<const uint4*>(scales + static_cast<size_t>(n) * G + 8 * b));
            const uint32_t* zp = zeros + static_cast<size_t>(n) * ZW + (8 * b) / PW;
            zblk[slot][0] = __ldg(zp);
            zblk[slot][1] = PW == 4 ? __ldg(zp + 1) : 0u;
          } else {
            sblk[slot] = make_uint4(0, 0, 0, 0);
            zblk[slot][0] = zblk[slot][1] = 0u;
          }
        };
        __half sq[kSzAhead];
        uint32_t zq[kSzAhead];
        auto load_sz = [&](int i, __half& sv, uint32_t& zv) {
          const int g = gfirst + i * gstride;
          if (row_ok && g < G) {
            sv = scales[static_cast<size_t>(n) * G + g];
            zv = (__ldg(zeros + static_cast<size_t>(n) * ZW + g / PW) >> ((g % PW) * BITS)) & QMASK;
          } else {
            sv = __ushort_as_half(0);
            zv = 0;
          }
        };
        const int gi0 = kb0 >> kb_shift;
        if (blocks8) {
          load_blk(gi0 >> 3, 0);
          load_blk((gi0 >> 3) + 1, 1);
        } else {
#pragma unroll
          for (int i = 0; i < kSzAhead; ++i) load_sz(gi0 + i, sq[i], zq[i]);
        }
        uint32_t zbe = 0x64006400u, zbo = 0x54005400u;
        __half2 s2 = __half2half2(__ushort_as_half(0));
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % S;
          if ((kb & kb_mask) == 0) {
            const int gi = kb >> kb_shift;   // this thread's group counter
            uint32_t zc;
            if (blocks8) {
              const int j = gi & 7;
              if (j == 0 && gi != gi0) {     // block done: the next one becomes current
                sblk[0] = sblk[1];
                zblk[0][0] = zblk[1][0];
                zblk[0][1] = zblk[1][1];
                load_blk((gi >> 3) + 1, 1);
              }
              const uint32_t sw = (j >> 1) == 0 ? sblk[0].x : (j >> 1) == 1 ? sblk[0].y
                                : (j >> 1) == 2 ? sblk[0].z : sblk[0].w;
              s2 = __half2half2(__ushort_as_half(static_cast<unsigned short>(sw >> (16 * (j & 1)))));
              zc = PW == 8 ? (zblk[0][0] >> (4 * j)) & QMASK
                           : (((j >> 2) == 0 ? zblk[0][0] : zblk[0][1]) >> (8 * (j & 3))) & QMASK;
            } else {
              s2 = __half2half2(sq[0]);
              zc = zq[0];
#pragma unroll
              for (int i = 0; i + 1 < kSzAhead; ++i) {
                sq[i] = sq[i + 1];
                zq[i] = zq[i + 1];
              }
              load_sz(gi + kSzAhead, sq[kSzAhead - 1], zq[kSzAhead - 1]);
            }
            zbe = (0x6400u | zc) * 0x00010001u;          // (1024 + z, 1024 + z)
            zbo = (0x5400u | (zc << 4)) * 0x00010001u;   // (64 + z, 64 + z), 4-bit only
          }
          if (!wait_or_abort(full + s, (it / S) & 1, ab, 4u)) {
            ok = false;
            break;
          }
          const uint8_t* rp = sRaw + s * C::RAW_BYTES + raw_r * C::RAW_ROW + half * (C::RAW_ROW / 2);
          uint8_t* arow = sA + s * C::A_BYTES + r * 128;
          if constexpr (BITS == 4) {
            const uint4 raw = *reinterpret_cast<const uint4*>(rp);
            const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int c = half * 4 + i;   // 16-byte chunk = 8 consecutive k
              *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) =
                  dequant_word<PERM>(rw[i], zbe, zbo, s2);
            }
          } else {
            const uint4 r0 = *reinterpret_cast<const uint4*>(rp);
            const uint4 r1 = *reinterpret_cast<const uint4*>(rp + 16);
            const uint32_t rw[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int c = half * 4 + i;   // 16-byte chunk = 8 consecutive k = 2 words
              *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) =
                  dequant_word8<PERM>(rw[2 * i], rw[2 * i + 1], zbe, s2);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(deq + s);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;   // TMEM lanes 32*quarter .. +31
    int lt = 0;
    for (int t = blockIdx.x; t < items; t += gridDim.x, ++lt) {
      int tile, kb0, kb1, split;
      item_of(t, tile, kb0, kb1, split);
      const int n0 = (tile % n_tiles) * BM, mt = tile / n_tiles, m0 = mt * BN;
      // a split tile's [BN][BM] block of partial sums for this part
      float* pout = split >= 0 ? part + (static_cast<size_t>(tile - full_tiles) * ts + split) *
                                            BN * BM
                               : nullptr;
      const int b = lt % C::ACC_BUFS;
      const int n = n0 + quarter * 32 + lane;
      if (!wait_or_abort(acc_full + b, (lt / C::ACC_BUFS) & 1, ab, 8u)) break;
      tc_fence_after();
      float sq = 0.f;
      for (int c0 = 0; c0 < BN; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + b * C::ACC_COLS + (static_cast<uint32_t>(quarter * 32) << 16) + c0, v);
        tmem_ld_wait();
        if constexpr (MODE == kGemmSiluF16) {
          // lanes 2i (gate) and 2i + 1 (up) hold one pair for 16 tokens; per
          // two tokens the gate lane finishes the first and the up lane the
          // second, after one exchange
          const int pair = n >> 1;
          const bool gate_lane = (lane & 1) == 0;
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const float a0 = __uint_as_float(v[j]), a1 = __uint_as_float(v[j + 1]);
            const float got = __shfl_xor_sync(0xffffffffu, gate_lane ? a1 : a0, 1);
            const float g = gate_lane ? a0 : got, u = gate_lane ? got : a1;
            const int m = m0 + c0 + j + (gate_lane ? 0 : 1);
            if (m < M && pair < N / 2)
              static_cast<__half*>(out)[static_cast<size_t>(m) * ldo + pair] =
                  __float2half_rn(g / (1.f + expf(-g)) * u);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = m0 + c0 + j;
            if (m < M && n < N) {
              const float val = __uint_as_float(v[j]);
              const size_t idx = static_cast<size_t>(m) * ldo + n;
              if (MODE == kGemmOutF16) {
                if (split >= 0)
                  pout[(m - m0) * BM + (n - n0)] = val;
                else
                  static_cast<__half*>(out)[idx] = __float2half_rn(val);
              } else if (MODE == kGemmDenseF32) {
                static_cast<float*>(out)[idx] = val;
              } else {
                const float e = val - yref[static_cast<size_t>(m) * ldy + n];
                sq = fmaf(e, e, sq);
              }
            }
          }
        }
      }
      if (MODE == kGemmSqErr && n < N)
        static_cast<float*>(out)[static_cast<size_t>(mt) * ldo + n] = sq;
      tc_fence_before();
      mbar_arrive(acc_empty + b);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// X~ = fp16(fp32(X) * inv_s), written with each 8-element chunk of k in the
// pair order the dequantization produces: (k0,k4) (k1,k5) (k2,k6) (k3,k7) for
// 4-bit codes, (k0,k2) (k1,k3) (k4,k6) (k5,k7) for 8-bit codes.
template <int BITS>
__global__ void prescale_kernel(const __half* __restrict__ X, const float* __restrict__ inv_s,
                                int64_t total8, int K, __half* __restrict__ Xt) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (i >= total8) return;
  const int k = static_cast<int>((i * 8) % K);
  const uint4 xr = __ldg(reinterpret_cast<const uint4*>(X) + i);
  const float4 a = __ldg(reinterpret_cast<const float4*>(inv_s + k));
  const float4 b = __ldg(reinterpret_cast<const float4*>(inv_s + k + 4));
  const float is[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  const __half* h = reinterpret_cast<const __half*>(&xr);
  uint4 o;
  __half2* oh = reinterpret_cast<__half2*>(&o);
  constexpr int lo[4] = {0, 1, BITS == 4 ? 2 : 4, BITS == 4 ? 3 : 5};
  constexpr int step = BITS == 4 ? 4 : 2;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int a0 = lo[j], a1 = lo[j] + step;
    oh[j] = __halves2half2(__float2half_rn(__fmul_rn(__half2float(h[a0]), is[a0])),
                           __float2half_rn(__fmul_rn(__half2float(h[a1]), is[a1])));
  }
  reinterpret_cast<uint4*>(Xt)[i] = o;
}

// The split tiles of the wide kernel: Y[m][n] = fp16(sum over s of the
// tile's part blocks, in order).  Tile full_tiles + tt, part s is the
// [bn][BM] block (tt * ts + s) of `part`.
__global__ void tile_reduce_kernel(const float* __restrict__ part, int full_tiles,
                                   int tail_tiles, int ts, int n_tiles, int bn, int M, int N,
                                   __half* __restrict__ Y, int ldo) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  constexpr int Q = BM / 4;   // float4 per block row
  const int64_t blk4 = static_cast<int64_t>(bn) * Q;   // float4 per [bn][BM] block
  const int64_t total = static_cast<int64_t>(tail_tiles) * blk4;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int tt = static_cast<int>(i / blk4);
    const int rem = static_cast<int>(i - tt * blk4);
    const int ml = rem / Q, n4 = rem - ml * Q;
    const int tile = full_tiles + tt;
    const int m = (tile / n_tiles) * bn + ml, n = (tile % n_tiles) * BM + 4 * n4;
    if (m >= M || n >= N) continue;
    const float4* src = reinterpret_cast<const float4*>(part) + tt * ts * blk4 + rem;
    float4 a = src[0];
    for (int s2 = 1; s2 < ts; ++s2) {
      const float4 b = src[s2 * blk4];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    __half2* y = reinterpret_cast<__half2*>(Y + static_cast<size_t>(m) * ldo + n);
    y[0] = __floats2half2_rn(a.x, a.y);
    y[1] = __floats2half2_rn(a.z, a.w);
  }
}

int launch_tile_reduce(const float* part, int full_tiles, int tail_tiles, int ts, int n_tiles,
                       int bn, int M, int N, __half* Y, int ldo, cudaStream_t st) {
  const int64_t total = static_cast<int64_t>(tail_tiles) * bn * (BM / 4);
  const int64_t want = (total + 255) / 256, cap = static_cast<int64_t>(sm_count()) * 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(want < cap ? want : cap), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  AWQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, tile_reduce_kernel, part, full_tiles, tail_tiles, ts,
                                  n_tiles, bn, M, N, Y, ldo));
  return AWQ_OK;
}

// Y[m][n] = fp16(sum over s of part[s][m][n]), the splits added in order.
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int splits, int64_t mn4,
                                     __half* __restrict__ Y) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < mn4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 a = reinterpret_cast<const float4*>(part)[i];
    for (int s = 1; s < splits; ++s) {
      const float4 b = reinterpret_cast<const float4*>(part)[s * mn4 + i];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    reinterpret_cast<__half2*>(Y)[2 * i] = __floats2half2_rn(a.x, a.y);
    reinterpret_cast<__half2*>(Y)[2 * i + 1] = __floats2half2_rn(a.z, a.w);
  }
}

template <int BN, int MODE, bool PERM, int BITS>
int launch_tile(const CUtensorMap& tb, const CUtensorMap& ta, const __half* scales,
                const uint32_t* zeros, int M, int N, int K, int gs, void* out, int ldo,
                const float* yref, int ldy, cudaStream_t st, int full_tiles = 0, int ts = 1,
                int kps = 0, float* part = nullptr) {
  using C = Cfg<BN, MODE, BITS>;
  if (kps == 0) kps = K / BK;
  {
    const int rc = ensure_smem_attr(reinterpret_cast<const void*>(gemm_kernel<BN, MODE, PERM, BITS>),
                                    C::SMEM);
    if (rc != AWQ_OK) return rc;
  }
  cudaLaunchConfig_t cfg = {};
  const int sms = sm_count();
  const int n_tiles = (N + BM - 1) / BM;
  const int tiles = n_tiles * ((M + BN - 1) / BN);
  const int items = full_tiles + (tiles - full_tiles) * ts;
  cfg.gridDim = dim3(items < sms ? items : sms, 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  AWQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, gemm_kernel<BN, MODE, PERM, BITS>, tb, ta, scales, zeros,
                                  M, N, K, gs, out, ldo, yref, ldy, full_tiles, ts, kps, part));
  if (ts > 1)
    return launch_tile_reduce(part, full_tiles, tiles - full_tiles, ts, n_tiles, BN, M, N,
                              static_cast<__half*>(out), ldo, st);
  return AWQ_OK;
}

template <int MODE, bool PERM, int BITS>
int dispatch_bn(int bn, const CUtensorMap& tb, const CUtensorMap& ta, const __half* scales,
                const uint32_t* zeros, int M, int N, int K, int gs, void* out, int ldo,
                const float* yref, int ldy, cudaStream_t st, int full_tiles, int ts, int kps,
                float* part) {
  switch (bn) {
    case 16:
      return launch_tile<16, MODE, PERM, BITS>(tb, ta, scales, zeros, M, N, K, gs, out, ldo, yref,
                                               ldy, st, full_tiles, ts, kps, part);
    case 32:
      return launch_tile<32, MODE, PERM, BITS>(tb, ta, scales, zeros, M, N, K, gs, out, ldo, yref,
                                               ldy, st, full_tiles, ts, kps, part);
    case 64:
      return launch_tile<64, MODE, PERM, BITS>(tb, ta, scales, zeros, M, N, K, gs, out, ldo, yref,
                                               ldy, st, full_tiles, ts, kps, part);
    case 128:
      return launch_tile<128, MODE, PERM, BITS>(tb, ta, scales, zeros, M, N, K, gs, out, ldo,
                                                yref, ldy, st, full_tiles, ts, kps, part);
    case 160:
      return launch_tile<160, MODE, PERM, BITS>(tb, ta, scales, zeros, M, N, K, gs, out, ldo,
                                                yref, ldy, st, full_tiles, ts, kps, part);
    default:
      return launch_tile<256, MODE, PERM, BITS>(tb, ta, scales, zeros, M, N, K, gs, out, ldo,
                                                yref, ldy, st, full_tiles, ts, kps, part);
  }
}

int pick_bn(int M, int mode) {
  if (mode != kGemmOutF16 && mode != kGemmSiluF16) return 256;
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 160;
}

}  // namespace

// Token-tile width and split-K for one launch.  The tile is the smallest of
// 16..256 tokens that holds M; the split comes from a cost model in SM
// cycles: a k-block of a work item costs max(2 BN, 208) cycles (tensor-core
// work of a 128 x BN x 64 MMA, or the 8 dequantization warps' share of 1024
// packed words, whichever is larger); items run in rounds of one per SM; a
// split pays its fp32 partial sums written and read back (8 bytes per output
// per part at ~3250 bytes per cycle) and a second launch.  Two kinds of split
// are weighed against none: every tile split s ways (for fewer tiles than
// SMs), and only the last, partial round of tiles split so that its parts
// fill the SMs that would otherwise idle while the other SMs run their
// whole tiles (for a few full rounds and a ragged one).  Only the plain fp16
// output splits (at most 8 parts of >= 8 k-blocks each).
GemmPlan plan_gemm(int M, int N, int K, int mode) {
  const int sms = sm_count();
  const int nk = K / BK;
  const int n_tiles = (N + BM - 1) / BM;
  // above 128 tokens the widest tile (measured: 128-token tiles lose more to
  // per-stage overheads than they win back on wave quantization)
  const int bn = pick_bn(M, mode);
  const int tiles = n_tiles * ((M + bn - 1) / bn);
  const double c = 2.0 * bn > 208.0 ? 2.0 * bn : 208.0;
  const double part_cost = 8.0 * bn * BM / 3250.0;   // per split tile and part
  GemmPlan best{bn, 0, 1, nk};
  double best_t = static_cast<double>((tiles + sms - 1) / sms) * nk * c;
  if (mode != kGemmOutF16) return best;
  const int rounds_full = tiles / sms, tail = tiles - rounds_full * sms;
  for (int s = 2; s <= 8; ++s) {
    const int kps = ((nk + s - 1) / s + 1) & ~1;
    if (kps < 8) break;
    if ((nk + kps - 1) / kps != s) continue;
    // every tile split
    {
      const int rounds = (tiles * s + sms - 1) / sms;
      const double t = static_cast<double>(rounds) * kps * c + part_cost * tiles * s + 2000.0;
      if (t < best_t) {
        best_t = t;
        best = GemmPlan{bn, 0, s, kps};
      }
    }
    // the ragged last round split, one part per otherwise idle SM
    if (rounds_full >= 1 && tail > 0 && tail * s <= sms) {
      const double t = (static_cast<double>(rounds_full) * nk + kps) * c + part_cost * tail * s +
                       2000.0;
      if (t < best_t) {
        best_t = t;
        best = GemmPlan{bn, rounds_full * sms, s, kps};
      }
    }
  }
  return best;
}

static size_t gemm_split_bytes(const GemmPlan& p, int M, int N) {
  if (p.ts <= 1) return 0;
  const int tiles = ((N + BM - 1) / BM) * ((M + p.bn - 1) / p.bn);
  return static_cast<size_t>(tiles - p.full_tiles) * p.ts * p.bn * BM * sizeof(float);
}

size_t gemm_partial_bytes(int M, int N, int K) {
  const size_t wide = gemm_split_bytes(plan_gemm(M, N, K, kGemmOutF16), M, N);
  const size_t narrow = narrow_partial_bytes(M, N, K);
  return wide > narrow ? wide : narrow;
}

int launch_splitk_reduce(const float* part, int splits, int M, int N, __half* Y,
                         cudaStream_t st) {
  const int64_t mn4 = static_cast<int64_t>(M) * N / 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sm_count() * 4), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  AWQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, part, splits, mn4, Y));
  return AWQ_OK;
}

int gemm_sqerr_slots(int M) { return (M + 255) / 256; }

int launch_prescale(const __half* X, const float* inv_s, int64_t M, int K, __half* Xt,
                    cudaStream_t st, int w_bit) {
  const int64_t total8 = M * K / 8;
  const int threads = 256;
  const int64_t blocks = (total8 + threads - 1) / threads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (w_bit == 8)
    AWQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, prescale_kernel<8>, X, inv_s, total8, K, Xt));
  else
    AWQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, prescale_kernel<4>, X, inv_s, total8, K, Xt));
  return AWQ_OK;
}

namespace {

template <int BITS>
int launch_gemm_bits(int mode, int bn, const CUtensorMap& tb, const CUtensorMap& ta,
                     bool xt_permuted, int M, const __half* scales, const uint32_t* zeros, int N,
                     int K, int gs, void* out, int ldo, const float* yref, int ldy,
                     cudaStream_t st, int full_tiles, int ts, int kps,
                     float* part) {
  switch (mode) {
    case kGemmOutF16:
      if (xt_permuted)
        return dispatch_bn<kGemmOutF16, true, BITS>(bn, tb, ta, scales, zeros, M, N, K, gs, out,
                                                    ldo, yref, ldy, st, full_tiles, ts, kps, part);
      return dispatch_bn<kGemmOutF16, false, BITS>(bn, tb, ta, scales, zeros, M, N, K, gs, out,
                                                   ldo, yref, ldy, st, full_tiles, ts, kps, part);
    case kGemmSiluF16:
      if constexpr (BITS == 4) {
        if (xt_permuted)
          return dispatch_bn<kGemmSiluF16, true, 4>(bn, tb, ta, scales, zeros, M, N, K, gs, out,
                                                    ldo, yref, ldy, st, 0, 1, 0, nullptr);
        return dispatch_bn<kGemmSiluF16, false, 4>(bn, tb, ta, scales, zeros, M, N, K, gs, out,
                                                   ldo, yref, ldy, st, 0, 1, 0, nullptr);
      }
      set_error("the fused gate/up layer takes 4-bit codes");
      return AWQ_ERR_UNSUPPORTED;
    case kGemmSqErr:
      if (!xt_permuted) {
        set_error("the squared-error matmul takes prescaled activations");
        return AWQ_ERR_UNSUPPORTED;
      }
      return launch_tile<256, kGemmSqErr, true, BITS>(tb, ta, scales, zeros, M, N, K, gs, out,
                                                      ldo, yref, ldy, st);
    default:
      return launch_tile<256, kGemmDenseF32, false, 4>(tb, ta, scales, zeros, M, N, K, gs, out,
                                                       ldo, yref, ldy, st);
  }
}

}  // namespace

int launch_gemm(int mode, const __half* Xt, bool xt_permuted, int M, const uint32_t* qweight,
                const __half* scales, const uint32_t* zeros, const __half* Wd, int N, int K,
                void* out, int ldo, const float* yref, int ldy, cudaStream_t st, int w_bit,
                int group, float* part, size_t part_bytes) {
  if ((w_bit != 4 && w_bit != 8) || (group != 32 && group != 64 && group != 128)) {
    set_error("awq_gemm: w_bit = %d, group = %d is not supported", w_bit, group);
    return AWQ_ERR_UNSUPPORTED;
  }
  if (mode == kGemmOutF16 && narrow_eligible(M, w_bit, group))
    return launch_gemm_narrow(Xt, xt_permuted, M, qweight, scales, zeros, N, K,
                              static_cast<__half*>(out), ldo, st, w_bit, group, part, part_bytes);
  GemmPlan plan = plan_gemm(M, N, K, mode);
  // a split needs the partial sums' workspace
  if (plan.ts > 1 &&
      (!part || part_bytes < gemm_split_bytes(plan, M, N) || !aligned16(part))) {
    plan.full_tiles = 0;
    plan.ts = 1;
    plan.kps = K / BK;
  }
  const int bn = plan.bn;
  CUtensorMap tb, ta;
  int rc = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Xt, K, M, static_cast<uint64_t>(K) * 2,
                        BK, bn, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != AWQ_OK) return rc;
  if (mode == kGemmSiluF16 && (N % 2 != 0)) {
    set_error("the fused gate/up weight needs an even number of rows");
    return AWQ_ERR_SHAPE;
  }
  if (mode == kGemmDenseF32) {
    rc = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Wd, K, N,
                      static_cast<uint64_t>(K) * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    const int pw = 32 / w_bit;       // codes per packed word
    // k-blocks per pipeline stage (Cfg::SK: 2 for the 160-token tile, whose
    // A operand is in tensor memory)
    const int sk = bn == 160 ? 2 : 1;
    rc = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT32, qweight, K / pw, N,
                      static_cast<uint64_t>(K / pw) * 4, sk * BK / pw,
                      mode == kGemmSiluF16 ? BM / 2 : BM, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (rc != AWQ_OK) return rc;
  if (w_bit == 8)
    return launch_gemm_bits<8>(mode, bn, tb, ta, xt_permuted, M, scales, zeros, N, K, group, out,
                               ldo, yref, ldy, st, plan.full_tiles, plan.ts, plan.kps, part);
  return launch_gemm_bits<4>(mode, bn, tb, ta, xt_permuted, M, scales, zeros, N, K, group, out,
                             ldo, yref, ldy, st, plan.full_tiles, plan.ts, plan.kps, part);
}

int set_gemm_stall(int withhold, uint64_t wait_ns) {
  const unsigned w = withhold ? 1u : 0u;
  const unsigned long long ns = wait_ns;
  AWQ_CUDA_TRY(cudaMemcpyToSymbol(g_gemm_withhold, &w, sizeof(w)));
  AWQ_CUDA_TRY(cudaMemcpyToSymbol(g_gemm_wait_ns, &ns, sizeof(ns)));
  return AWQ_OK;
}

int read_clear_gemm_error(cudaStream_t st, unsigned* flags) {
  AWQ_CUDA_TRY(cudaStreamSynchronize(st));
  unsigned v = 0, zero = 0;
  AWQ_CUDA_TRY(cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(v)));
  AWQ_CUDA_TRY(cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(zero)));
  *flags = v;
  return AWQ_OK;
}

}  // namespace awq
