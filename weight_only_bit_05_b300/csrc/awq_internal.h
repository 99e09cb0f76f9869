// Internal launchers behind the C ABI (C++ linkage, one per translation unit).
// Arguments are already validated by the entry points in awq_api.cu.
#pragma once

#include "awq_common.cuh"

namespace awq {

// awq_api.cu: per-device launch helpers, safe to call from several host
// threads.  sm_count: SMs of the current device (148 when it cannot be
// queried).  ensure_smem_attr: raises the kernel's dynamic shared-memory limit
// on the current device to at least `bytes` (once per kernel and device).
int sm_count();
int ensure_smem_attr(const void* func, int bytes);

// awq_stats.cu
size_t absmean_workspace_size(int64_t T, int K);
int launch_absmean(const __half* X, int64_t T, int K, float* a, void* ws, cudaStream_t st);
int launch_channel_scales(const float* a, int K, double alpha, float* s_c, float* inv_s,
                          cudaStream_t st);

// awq_pack.cu
// w_bit 4 or 8, group 128/64/32, zero_point on (asymmetric) or off
// (symmetric: codes offset by 2^(w_bit-1), stored as the zero point).
// clip_idx (optional, uint8 [N][G]) shrinks each group's range by the ratio
// 1 - 0.5 i / n_clip before quantization.
int launch_pack(const __half* W, const float* s_c, int N, int K, uint32_t* qweight,
                __half* scales, uint32_t* zeros, cudaStream_t st, int w_bit = 4,
                int group = 128, bool zero_point = true, const uint8_t* clip_idx = nullptr,
                int n_clip = 1);

// Empty non-PDL kernel ending the entry points that write packed weights.
int launch_stream_fence(cudaStream_t st);

// awq_clip.cu
size_t clip_workspace_size(int64_t T, int K, int group);
int launch_clip_search(const __half* X, int64_t T, const __half* W, int N, int K,
                       const float* s_c, const float* inv_s, int w_bit, int group,
                       bool zero_point, int n_clip, void* ws, uint8_t* clip_idx, float* err,
                       cudaStream_t st);

// awq_gemv.cu
// silu_mul: the weight's N rows are I = N/2 gate rows over I up rows and Y
// receives silu(gate) * up, [M][N/2].
// w_bit 4 or 8 and group 128/64/32 give the packed layout (silu_mul: 4/128).
int launch_gemv(const __half* X, int M, const uint32_t* qweight, const __half* scales,
                const uint32_t* zeros, const float* inv_s, int N, int K, __half* Y,
                cudaStream_t st, bool silu_mul = false, int w_bit = 4, int group = 128);

// awq_gemv_mma.cu: the decode matmul for 4-bit codes in 128-channel groups,
// M <= 8, K % 256 == 0 (weights streamed by TMA before the dependency wait,
// dot products on the warp-level MMA).
struct MmaGemvPlan {
  int warps;         // warps per CTA, each with its own ring of stages
  int depth;         // stages per warp ring (0: no plan fits)
  int nsplit;        // K slices (thread-block cluster size along y)
  int KS;            // input channels per slice
  int gx;            // CTAs along the rows
  int rows_cap;      // most rows of one CTA
  int smem;          // dynamic shared memory per CTA
  int ctas_per_sm;   // CTAs of one launch per SM (1 or 2)
};
MmaGemvPlan plan_gemv_mma(int M, int N, int K, int sms);
MmaGemvPlan make_gemv_mma_plan(int M, int N, int K, int sms, int warps, int ctas_per_sm,
                               int min_depth, int max_depth);
int launch_gemv_mma_plan(const MmaGemvPlan& p, const __half* X, int M, const uint32_t* qweight,
                         const __half* scales, const uint32_t* zeros, const float* inv_s, int N,
                         int K, __half* Y, cudaStream_t st);
bool gemv_mma_eligible(int M, int K, int w_bit, int group, bool silu_mul);
int launch_gemv_mma(const __half* X, int M, const uint32_t* qweight, const __half* scales,
                    const uint32_t* zeros, const float* inv_s, int N, int K, __half* Y,
                    cudaStream_t st);
int read_clear_gemv_error(cudaStream_t st, unsigned* flags);
// Test hook of the decode matmul's bounded waits (device-wide, current device).
int set_gemv_stall(int withhold, uint64_t wait_ns);

// awq_measure.cu: streaming read of `bytes` (a multiple of 16) for the
// bandwidth ceiling of a chain of launches; `out` receives nothing unless the
// buffer folds to one particular word (one word per SM must be writable).
int launch_stream_read(const void* buf, size_t bytes, int read_first, unsigned* out,
                       cudaStream_t st);

// awq_fold.cu
int launch_fold_inv_scales(const __half* W, int64_t rows, int64_t cols, const float* inv_s,
                           __half* out, cudaStream_t st);

// awq_gemm.cu
enum GemmMode { kGemmOutF16 = 0, kGemmSqErr = 1, kGemmDenseF32 = 2, kGemmSiluF16 = 3 };
// Xt = fp16(X * inv_s), each 8-element chunk of k stored in the pair order of
// the dequantization of w_bit-bit codes ((k0,k4) (k1,k5) (k2,k6) (k3,k7) for 4,
// (k0,k2) (k1,k3) (k4,k6) (k5,k7) for 8): the layout launch_gemm takes with
// xt_permuted = true.
int launch_prescale(const __half* X, const float* inv_s, int64_t M, int K, __half* Xt,
                    cudaStream_t st, int w_bit = 4);
// Runs the tensor-core kernel on activations `Xt` [M][K] (already scaled;
// xt_permuted says whether k is in the prescale kernel's chunk order, which
// the quantized modes prefer, or natural).
//   kGemmOutF16  : Y = fp16(Xt * dequant(qweight)^T), out = fp16 [M][ldo]
//   kGemmSqErr   : out = fp32 partial sums of (Xt*dequant^T - yref)^2 per
//                  output row, [ceil(M/256)*2][ldo]; yref fp32 [M][ldy]
//   kGemmDenseF32: out = fp32 Xt * Wd^T, Wd fp16 [N][K] dense
//   kGemmSiluF16 : the N weight rows stack N/2 gate rows over N/2 up rows;
//                  out = fp16 silu(gate) * up, [M][ldo] with N/2 columns
// part/part_bytes: workspace for split-K partial sums (kGemmOutF16 only; with
// too little or none the launch runs without split-K).
int launch_gemm(int mode, const __half* Xt, bool xt_permuted, int M, const uint32_t* qweight,
                const __half* scales, const uint32_t* zeros, const __half* Wd, int N, int K,
                void* out, int ldo, const float* yref, int ldy, cudaStream_t st, int w_bit = 4,
                int group = 128, float* part = nullptr, size_t part_bytes = 0);
struct GemmPlan {
  int bn;           // token-tile width
  int full_tiles;   // tiles 0 .. full_tiles - 1 run whole
  int ts;           // the rest are split over K, ts ways each (1: no split)
  int kps;          // k-blocks (64 channels) per split
};
GemmPlan plan_gemm(int M, int N, int K, int mode);
size_t gemm_partial_bytes(int M, int N, int K);   // split-K workspace of the plain matmul
int gemm_sqerr_slots(int M);   // number of partial rows kGemmSqErr writes
int read_clear_gemm_error(cudaStream_t st, unsigned* flags);
// Test hook of the wide tensor-core matmul's bounded waits (current device).
int set_gemm_stall(int withhold, uint64_t wait_ns);
// Y[m][n] = fp16(sum over s < splits of part[s][m][n]), part fp32 [splits][M][N].
int launch_splitk_reduce(const float* part, int splits, int M, int N, __half* Y,
                         cudaStream_t st);

// awq_gemm_narrow.cu: the plain fp16-output matmul for M <= 128 tokens, 4- or
// 8-bit codes in 128- or 64-channel groups (per-group tensor-memory
// accumulators, steps applied in fp32 by the epilogue).
constexpr int kNarrowMaxM = 128;
struct NarrowPlan {
  int bn;       // token-tile width (0: not eligible)
  int splits;   // split-K factor
  int kps;      // stages per split
  int bks;      // input channels per stage
};
bool narrow_eligible(int M, int w_bit, int group);
NarrowPlan plan_narrow(int M, int N, int K, int w_bit, int group);
size_t narrow_partial_bytes(int M, int N, int K);   // split-K workspace, any eligible format
int launch_gemm_narrow(const __half* Xt, bool xt_permuted, int M, const uint32_t* qweight,
                       const __half* scales, const uint32_t* zeros, int N, int K, __half* out,
                       int ldo, cudaStream_t st, int w_bit, int group, float* part,
                       size_t part_bytes);
int read_clear_narrow_error(cudaStream_t st, unsigned* flags);

}  // namespace awq
