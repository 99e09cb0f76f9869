/*
 * awq.h - C ABI of the B300 (sm_103a) AWQ W4A16 group-quantized linear layer.
 *
 * The method (Activation-aware Weight Quantization) as described by the pages
 * "AWQ量化实战：无需重训，把大模型压进4bit显存" (§2.1-§2.3, §3.3),
 * "大模型量化部署实战：GPTQ与AWQ算法" (section 大模型量化的核心原理与位宽选择)
 * and "什么是激活感知权重量化（AWQ）？" (section 工作机制):
 *
 *   a_c    = mean_t |x_tc|                       per input channel (statistics)
 *   s_c    = a_c ^ alpha,  alpha in {0, 1/20, ..., 19/20}
 *   W'     = W diag(s_c)                          equivalent transformation
 *   per (row n, group g of 128 input channels):   asymmetric round-to-nearest
 *     s = fp16((max - min) / 15) clamped to [2^-14, 65504],
 *     z = clamp(rint(-min / s), 0, 15),  q = clamp(rint(w' / s) + z, 0, 15)
 *   w^'    = (q - z) * s                          dequantization
 *   Y      = (X diag(1/s_c)) W^'^T                the quantized linear layer
 *   alpha* = argmin over the grid of mean((Y - X W^T)^2) on calibration tokens
 *
 * Conventions for every entry point
 *   - Matrices are row-major and dense. W is [N][K]: row n is output channel n,
 *     column k is input channel k. X is [M][K] (tokens x input channels).
 *   - fp16 data is passed as uint16_t bit patterns (IEEE binary16).
 *   - Unless stated otherwise every pointer is a DEVICE pointer on the current
 *     CUDA device, owned by the caller; the library never frees it and keeps no
 *     reference after the call. Every device pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *     asynchronous on that stream unless stated otherwise.
 *   - Shapes: K % 128 == 0, N % 8 == 0, M >= 1. The return value is a status
 *     code below; on failure nothing was launched and
 *     awq_last_error_string() (thread-local) says why.
 *   - The library allocates no device memory on its own: kernels that need
 *     scratch take a caller-provided workspace whose size the matching
 *     *_workspace_size() function returns.
 *
 * Canonical packed layout (the library's own; the pages only name
 * "platform-aware weight packing", "什么是激活感知权重量化（AWQ）？" 典型例子), for the
 * default configuration (4-bit codes, 128-channel groups; other configurations
 * at awq_config below):
 *   qweight uint32 [N][K/8]        : word j of row n holds k = 8j+i in bits [4i, 4i+4)
 *   scales  fp16   [N][K/128]      : step of group g of row n
 *   zeros   uint32 [N][ceil(G/8)]  : group g = 8j+i in bits [4i, 4i+4); unused nibbles 0
 */
#ifndef AWQ_H_
#define AWQ_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define AWQ_API __attribute__((visibility("default")))
#else
#define AWQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define AWQ_OK              0
#define AWQ_ERR_SHAPE       1  /* K % 128, N % 8, M or T out of range */
#define AWQ_ERR_NULL        2  /* a required pointer is NULL */
#define AWQ_ERR_ALIGN       3  /* a device pointer is not 16-byte aligned */
#define AWQ_ERR_CUDA        4  /* a CUDA runtime/driver call failed */
#define AWQ_ERR_UNSUPPORTED 5  /* configuration not implemented (w_bit, group, zero_point) */
#define AWQ_ERR_WORKSPACE   6  /* workspace NULL, too small or misaligned */
#define AWQ_ERR_DEVICE      7  /* a kernel reported a bounded wait that ran out */

/* Quantization configuration ("awq-quantization" skill page, 步骤 2: zero_point,
 * q_group_size, w_bit). w_bit 4 or 8 ("AWQ量化实战" §3.3: 8 bits as the
 * conservative width), group 128, 64 or 32 (§2.3), zero_point 1 (asymmetric) or
 * 0 (symmetric, §3.3; "大模型量化部署实战" gives the signed int4 range -8..7);
 * n_grid is the number of alpha candidates (1..64, default 20).
 * Packed layout for a configuration (c = 32 / w_bit codes per word, G = K/group):
 *   qweight uint32 [N][K/c]      : word j of row n holds k = c j + i in bits [w_bit i, w_bit (i+1))
 *   scales  fp16   [N][G]        : step of group g of row n
 *   zeros   uint32 [N][ceil(G/c)]: group g = c j + i in field i; unused fields 0
 * Symmetric codes are stored offset by h = 2^(w_bit-1) (q = clamp(rint(w'/s),
 * -h, h-1) + h with s = max|w'| / (h-1)), and every zero point is h, so the
 * matmuls dequantize every configuration as (q - z) * s. */
typedef struct awq_config {
  int32_t w_bit;
  int32_t group;
  int32_t zero_point;
  int32_t n_grid;
} awq_config;

/* Default configuration {4, 128, 1, 20}. */
AWQ_API awq_config awq_default_config(void);

/* Human-readable reason of the last failing call on this host thread. */
AWQ_API const char* awq_last_error_string(void);

/* Reads and clears the device-side error words of the kernels that use
 * bounded waits (the tensor-core matmuls and the decode matmul): every wait on
 * an mbarrier gives up after a limit (1 s) instead of hanging, records the
 * fact in a word of the current device, lets its copies in flight land and
 * returns; the output of that call is then undefined. The words are per
 * device and shared by all streams and host threads, so this call first
 * synchronizes the whole current device (`stream` is not used beyond that)
 * and reports a timeout of any call on the device since the last check.
 * Returns AWQ_OK if none, AWQ_ERR_DEVICE otherwise. */
AWQ_API int awq_check_device_error(void* stream);

/* ---------------------------------------------------------------- statistics
 * a[c] = (1/T) * sum_t |X[t][c]|   ("AWQ量化实战" §2.1: mean absolute activation
 * of each input channel over the calibration tokens).
 * X: fp16 [T][K] device. a: fp32 [K] device (output).
 * Sums are fp32 over runs of 16 tokens, then fp64; the result is
 * deterministic (fixed reduction order).
 * workspace: device, >= awq_absmean_workspace_size(T, K) bytes, 16-B aligned. */
AWQ_API size_t awq_absmean_workspace_size(int64_t T, int32_t K);
AWQ_API int awq_absmean(const uint16_t* X, int64_t T, int32_t K, float* a,
                void* workspace, size_t ws_bytes, void* stream);

/* Same statistics as awq_absmean for callers that cannot provide device memory:
 * runtimes that plan every buffer before execution and forbid allocation on the
 * execution path, real-time loops where an allocation's latency or failure is
 * not acceptable, plugins whose host framework owns all device memory. The pages
 * have no counterpart of this entry point; it exists for such callers only.
 * The partial sums live in a fixed 4 MiB array of device memory inside the
 * library, which every GPU that loads the library holds until the process
 * exits. K is limited to 524288 input channels (larger K returns
 * AWQ_ERR_SHAPE); T is not limited. The first call on a device looks up the
 * array's device address on that device (call it once before any stream
 * capture). Every call shares the one array: calls that overlap on the GPU
 * (other streams, other threads) race and give wrong results; serialize them.
 * No memory is allocated or freed by this call. X: fp16 [T][K], a: fp32 [K]. */
AWQ_API int awq_absmean_noalloc(const uint16_t* X, int64_t T, int32_t K, float* a,
                                void* stream);

/* ----------------------------------------------------------- channel scales
 * s_c[k] = fp32(pow(fp64(max(a[k], 1e-8f)), alpha)), inv_s[k] = 1.0f / s_c[k]
 * (IEEE fp32 division). alpha must lie in [0, 1).
 * ("AWQ量化实战" §2.2: salient channels are scaled up by a factor taken from the
 * activation statistics.) a, s_c, inv_s: fp32 [K] device. */
AWQ_API int awq_channel_scales(const float* a, int32_t K, double alpha, float* s_c,
                       float* inv_s, void* stream);

/* ---------------------------------------------------------------- quantizer
 * Scaled group RTN and packing into the canonical layout of the configuration
 * ("AWQ量化实战" §1.1, §2.3, §3.3; "大模型量化部署实战" 核心原理). Codes are decided
 * in fp32 with IEEE division and round-half-even, bit-exact with the definition.
 * W: fp16 [N][K]. s_c: fp32 [K] or NULL (all ones). cfg: NULL = 4/128/1.
 * Default layout: qweight uint32 [N][K/8]; scales fp16 [N][K/128]; zeros uint32
 * [N][ceil(G/8)]; other configurations as described at awq_config. */
AWQ_API int awq_pack(const uint16_t* W, const float* s_c, int32_t N, int32_t K,
             const awq_config* cfg, uint32_t* qweight, uint16_t* scales,
             uint32_t* zeros, void* stream);

/* ------------------------------------------------------------ GEMV, M <= 8
 * Y[m][n] = fp16( sum_k (X[m][k] * inv_s[k]) * (q[n][k] - z[n][g(k)]) * s[n][g(k)] )
 * ("awq-quantization" skill page, 主要功能: the GEMV kernel serves batch-1
 * token generation; "AWQ量化实战" §3.4: decoding is bound by reading the
 * weights.)  X: fp16 [M][K], 1 <= M <= 8. inv_s: fp32 [K] or NULL (all
 * ones). Y: fp16 [M][N]. The result is deterministic.
 * The default format (4-bit codes, 128-channel groups) with K % 256 == 0
 * streams the packed codes, steps and zero points through TMA and cp.async
 * into shared memory and reduces on the warp-level tensor-core MMA (exact
 * products x~ (q - z), fp32 sums, each group's sum times its step in fp32);
 * other formats and K run on CUDA cores (fp32 products and sums,
 * warp-shuffle reductions). K is split over a thread-block cluster when the
 * activations do not fit in shared memory.
 * Launched with programmatic dependent launch: qweight, scales and zeros are
 * read BEFORE the kernel waits for the previous kernel on the stream, so that
 * the weights of consecutive layers stream without a gap. They must therefore
 * not be written by the kernel launched immediately before this call on the
 * same stream (awq_pack and awq_pack_clipped end with an empty kernel for
 * this reason, so calling awq_gemv right after them is safe). X, inv_s and Y
 * are touched only after the wait. */
AWQ_API int awq_gemv(const uint16_t* X, int32_t M, const uint32_t* qweight,
             const uint16_t* scales, const uint32_t* zeros, const float* inv_s,
             int32_t N, int32_t K, uint16_t* Y, void* stream);

/* awq_gemv for a configuration's packed layout (cfg NULL = the default 4/128/1;
 * zero_point does not matter to the matmul, the zero points are stored). */
AWQ_API int awq_gemv_ex(const awq_config* cfg, const uint16_t* X, int32_t M,
                const uint32_t* qweight, const uint16_t* scales, const uint32_t* zeros,
                const float* inv_s, int32_t N, int32_t K, uint16_t* Y, void* stream);

/* ------------------------------------------------------------- GEMM, any M
 * Same result as awq_gemv for any M >= 1. For M <= 8 with the default format
 * (K % 256 == 0) it runs awq_gemv's decode matmul whenever that needs no K
 * split or halves K over a cluster of two (the workspace is then unused).
 * Otherwise on the 5th-generation
 * tensor cores:
 * packed codes and activations staged by TMA, codes dequantized to fp16
 * (into tensor memory for the tcgen05.mma's A operand above 128 tokens,
 * into shared memory otherwise), tcgen05.mma (fp16 x fp16, fp32
 * accumulation in tensor memory). For M <= 128 with 4- or 8-bit codes in
 * 128- or 64-channel groups
 * a narrow-token kernel runs instead: the operand holds the exact integers
 * q - z in tensor memory, each group's partial sum is accumulated on its own
 * and multiplied by the group step in fp32 (so it rounds differently from
 * the wide kernel, within the same bound). ("awq-quantization" skill page,
 * 主要功能: the GEMM kernel serves batch > 1.) When inv_s is not NULL,
 * X~ = fp16(X * inv_s) is first written
 * to the workspace; with inv_s == NULL X is read directly and the workspace
 * may be NULL. awq_gemm_workspace_size also counts the fp32 partial sums of a
 * split-K launch, chosen either when the layer has too few 128-row tiles to
 * fill the GPU (every tile split over K) or when the tiles fill a few rounds
 * of the SMs and leave a ragged last one (only that round's tiles split, so
 * their parts occupy the SMs that would idle); a second kernel adds each
 * tile's parts in a fixed order. A smaller workspace, at least X~ when inv_s
 * is given, runs without split-K.
 * Y: fp16 [M][N]. */
AWQ_API size_t awq_gemm_workspace_size(int32_t M, int32_t N, int32_t K);
AWQ_API int awq_gemm(const uint16_t* X, int32_t M, const uint32_t* qweight,
             const uint16_t* scales, const uint32_t* zeros, const float* inv_s,
             int32_t N, int32_t K, uint16_t* Y, void* workspace,
             size_t ws_bytes, void* stream);
/* awq_gemm for a configuration's packed layout (cfg NULL = 4/128/1); the
 * workspace rule is the same. */
AWQ_API int awq_gemm_ex(const awq_config* cfg, const uint16_t* X, int32_t M,
                const uint32_t* qweight, const uint16_t* scales, const uint32_t* zeros,
                const float* inv_s, int32_t N, int32_t K, uint16_t* Y, void* workspace,
                size_t ws_bytes, void* stream);

/* ------------------------------------------ fused gate/up (MLP) projection
 * The two projections of an MLP that read the same input run as one layer
 * ("awq-quantization" skill page, 主要功能和特点: fused attention/MLP modules;
 * "什么是激活感知权重量化（AWQ）？": kernel fusion in TinyChat). The weight is the
 * stack [gate; up] of 2I rows, packed, searched and scaled as one [2I][K]
 * layer (one s_c for both, since both read the same activations):
 *   Y[m][j] = fp16( silu(g_mj) * u_mj ),  silu(x) = x / (1 + exp(-x)),
 * where g_mj and u_mj are the fp32 sums of awq_gemv/awq_gemm for rows j and
 * I + j, formed in registers without an fp16 rounding in between.
 * X: fp16 [M][K]; qweight/scales/zeros: [2I] rows of the canonical layout;
 * inv_s: fp32 [K] or NULL; Y: fp16 [M][I]. I % 4 == 0, K % 128 == 0.
 * awq_gemv_silu_mul takes 1 <= M <= 8 (CUDA cores, as awq_gemv);
 * awq_gemm_silu_mul any M >= 1 (tensor cores, as awq_gemm, same workspace
 * rule: awq_gemm_workspace_size(M, 2I, K) bytes when inv_s is not NULL). */
AWQ_API int awq_gemv_silu_mul(const uint16_t* X, int32_t M, const uint32_t* qweight,
                      const uint16_t* scales, const uint32_t* zeros,
                      const float* inv_s, int32_t I, int32_t K, uint16_t* Y,
                      void* stream);
AWQ_API int awq_gemm_silu_mul(const uint16_t* X, int32_t M, const uint32_t* qweight,
                      const uint16_t* scales, const uint32_t* zeros,
                      const float* inv_s, int32_t I, int32_t K, uint16_t* Y,
                      void* workspace, size_t ws_bytes, void* stream);

/* ----------------------------- the equivalent transformation, folded offline
 * ("什么是激活感知权重量化（AWQ）？", 工作机制: salient channels are protected by an
 * equivalent transformation whose factors come from offline activation
 * statistics.) (x diag(1/s_c)) (W diag(s_c))^T = x W^T, so 1/s_c can be moved
 * into the operator that produces x instead of being applied at run time
 * (then pass inv_s = NULL to the matmuls):
 *   out[r][c] = fp16( fp32(W[r][c]) * inv_s[r] )   (one rounding, to nearest)
 * W: fp16 [rows][cols], one row per input channel of the quantized layer: a
 * norm's weight vector (rows = K, cols = 1) or the output rows of the previous
 * linear ([K][C]). inv_s: fp32 [rows]. out may equal W (in place).
 * rows >= 1, cols >= 1. */
AWQ_API int awq_fold_inv_scales(const uint16_t* W, int64_t rows, int64_t cols,
                        const float* inv_s, uint16_t* out, void* stream);

/* ---------------------------------------------------- weight clipping
 * ("AWQ量化实战" §5.1 names a clipping parameter, clip_steps, suggested 200,
 * and nothing more.)  Library reading: after the scale search, each group's
 * range [min, max] of the scaled weights W diag(s_c) may shrink to
 * [r min, r max] (symmetric: r max|w'|) with r_i = fp32(1 - 0.5 i / n_clip),
 * i = 0 .. n_clip-1; the group is quantized from the shrunk range (codes clamp,
 * which clips) and the ratio with the smallest output error on the calibration
 * tokens, d^T H_g d with d = w^ - w' and H_g = X~_g^T X~_g (x~ = x * inv_s),
 * is kept; ties go to the least clipping (smallest i).
 * awq_clip_search: X_cal fp16 [T][K]; W fp16 [N][K]; s_c, inv_s fp32 [K] or
 * NULL (the scales of the chosen alpha); clip_idx out uint8 [N][G] device;
 * err_out fp32 [N][G][n_clip] device or NULL (every candidate's error, fp32
 * sums); 1 <= n_clip <= 200. Workspace: awq_clip_search_workspace_size bytes
 * (the group Gram matrices and their per-chunk partial sums).
 * awq_pack_clipped: awq_pack with each group's range shrunk by
 * clip_idx[n][g] (n_clip as in the search); clip_idx all 0 is awq_pack. */
AWQ_API size_t awq_clip_search_workspace_size(int64_t T, int32_t K, const awq_config* cfg);
AWQ_API int awq_clip_search(const uint16_t* X_cal, int64_t T, const uint16_t* W,
                    int32_t N, int32_t K, const float* s_c, const float* inv_s,
                    const awq_config* cfg, int32_t n_clip, void* workspace,
                    size_t ws_bytes, uint8_t* clip_idx, float* err_out, void* stream);
AWQ_API int awq_pack_clipped(const uint16_t* W, const float* s_c, int32_t N, int32_t K,
                     const awq_config* cfg, const uint8_t* clip_idx, int32_t n_clip,
                     uint32_t* qweight, uint16_t* scales, uint32_t* zeros,
                     void* stream);

/* ------------------------------------------------------------ scale search
 * The activation-aware grid search ("AWQ量化实战" §2.2, §3.3 第四步, §5.1: one
 * coefficient per layer, no backpropagation): a = absmean(X_cal); for each
 * alpha_i = i / n_grid: s_c = a^alpha_i, quantize W diag(s_c), run the
 * quantized layer on the calibration tokens on the tensor cores and reduce
 * mse_i = sum (Y^ - X_cal W^T)^2 / (T N) (fp32 per tile, fp64 across tiles).
 * alpha* = first index of the smallest mse.
 * X_cal: fp16 [T][K]; W: fp16 [N][K]; s_c_out, inv_s_out: fp32 [K] device
 * (scales of the chosen alpha); best_out: HOST int32 (index of alpha*);
 * mse_out: HOST double [n_grid]; row_err_out: DEVICE double [n_grid][N] or
 * NULL (per-output-row squared error sums, for validation).
 * Synchronizes `stream` (the host reads the n_grid errors). */
AWQ_API size_t awq_search_workspace_size(int64_t T, int32_t N, int32_t K);
AWQ_API int awq_search_scales(const uint16_t* X_cal, int64_t T, const uint16_t* W,
                      int32_t N, int32_t K, const awq_config* cfg,
                      void* workspace, size_t ws_bytes, float* s_c_out,
                      float* inv_s_out, int32_t* best_out, double* mse_out,
                      double* row_err_out, void* stream);

/* --------------------------------------------------------------- test hook
 * Not a step of the method (the pages have no counterpart): lets a test drive
 * the bounded waits to expiry without faulting or hanging the GPU.
 * `which` selects the kernels whose following launches on the current device
 * lose one copy: bit 0 (1) the decode matmul of awq_gemv's default format
 * (the first CTA does not request its first stage), bit 1 (2) the
 * wide tensor-core matmul of awq_gemm, M > 128 (the producer of the first CTA
 * does not request its first stage). The wait for that stage runs out after
 * wait_limit_ns, the kernel records it for awq_check_device_error, stops its
 * other roles, waits (bounded) for its copies and MMAs in flight, frees its
 * tensor memory and returns; that call's Y is undefined. wait_limit_ns (1e3 ..
 * 1e10) becomes the limit of every bounded wait of both kernels.
 * awq_debug_stall(0, 1000000000) restores the defaults. Device-wide state:
 * not for concurrent use. */
AWQ_API int awq_debug_stall(int32_t which, int64_t wait_limit_ns);

/* --------------------------------------------------------- measurement aid
 * Not a step of the method (the pages have no counterpart): a plain streaming
 * read of `bytes` bytes at `buf` (device, 16-byte aligned, bytes a multiple of
 * 16), launched like awq_gemv with programmatic dependent launch, one CTA per
 * SM. A chain of these over the same weight buffers as a chain of awq_gemv
 * calls measures the bandwidth ceiling that HBM and the overlap of
 * consecutive launches leave such a chain. read_first != 0 issues the reads
 * before waiting for the previous kernel in the stream (as awq_gemv does with
 * its weights), 0 after. `out`: device, one uint32 per SM, written only when
 * the buffer's words fold to one particular value. */
AWQ_API int awq_measure_stream_read(const void* buf, size_t bytes, int32_t read_first,
                                    uint32_t* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif  /* AWQ_H_ */
