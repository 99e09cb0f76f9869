// C-ABI entry points: argument validation, status codes and error strings.
// Every step of the computation runs in the kernels of the other files.
#include <atomic>
#include <cstdarg>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "awq_internal.h"

namespace awq {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return AWQ_OK;
  set_error("%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  return AWQ_ERR_CUDA;
}

// ------------------------------------------------ per-device launch helpers
// A process may drive several devices from several host threads: the SM
// count is cached per device ordinal, and the dynamic shared-memory limit of
// a kernel is raised once per (kernel, device) under a lock.
namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];
std::mutex g_attr_mu;
std::map<std::pair<const void*, int>, int> g_attr_bytes;
}  // namespace

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  int n = g_sms[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  g_sms[dev].store(n, std::memory_order_relaxed);
  return n;
}

int ensure_smem_attr(const void* func, int bytes) {
  int dev = 0;
  AWQ_CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(g_attr_mu);
  int& have = g_attr_bytes[std::make_pair(func, dev)];
  if (have >= bytes) return AWQ_OK;
  AWQ_CUDA_TRY(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
  have = bytes;
  return AWQ_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t cols,
                 uint64_t rows, uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows,
                 CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the CUDA driver");
    return AWQ_ERR_CUDA;
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (CUresult %d) for %llux%llu box %ux%u",
              static_cast<int>(r), (unsigned long long)rows, (unsigned long long)cols, box_rows,
              box_cols);
    return AWQ_ERR_CUDA;
  }
  return AWQ_OK;
}

}  // namespace awq

using namespace awq;

namespace {

int check_kn(int32_t N, int32_t K) {
  if (K <= 0 || K % kGroup != 0) {
    set_error("K = %d must be a positive multiple of 128", K);
    return AWQ_ERR_SHAPE;
  }
  if (N <= 0 || N % 8 != 0) {
    set_error("N = %d must be a positive multiple of 8", N);
    return AWQ_ERR_SHAPE;
  }
  return AWQ_OK;
}

int check_ptr(const void* p, const char* name) {
  if (!p) {
    set_error("%s is NULL", name);
    return AWQ_ERR_NULL;
  }
  if (!aligned16(p)) {
    set_error("%s is not 16-byte aligned", name);
    return AWQ_ERR_ALIGN;
  }
  return AWQ_OK;
}

int check_opt_ptr(const void* p, const char* name) { return p ? check_ptr(p, name) : AWQ_OK; }

int check_cfg(const awq_config* cfg) {
  if (!cfg) return AWQ_OK;  // NULL means the default configuration
  if ((cfg->w_bit != 4 && cfg->w_bit != 8) ||
      (cfg->group != 128 && cfg->group != 64 && cfg->group != 32) ||
      (cfg->zero_point != 0 && cfg->zero_point != 1)) {
    set_error("unsupported configuration w_bit=%d group=%d zero_point=%d (w_bit 4 or 8, "
              "group 128, 64 or 32, zero_point 0 or 1)", cfg->w_bit, cfg->group, cfg->zero_point);
    return AWQ_ERR_UNSUPPORTED;
  }
  if (cfg->n_grid < 1 || cfg->n_grid > 64) {
    set_error("n_grid = %d must be in [1, 64]", cfg->n_grid);
    return AWQ_ERR_UNSUPPORTED;
  }
  return AWQ_OK;
}

#define AWQ_TRY(x)               \
  do {                           \
    int _s = (x);                \
    if (_s != AWQ_OK) return _s; \
  } while (0)

}  // namespace

extern "C" {

awq_config awq_default_config(void) {
  awq_config c;
  c.w_bit = 4;
  c.group = 128;
  c.zero_point = 1;
  c.n_grid = 20;
  return c;
}

const char* awq_last_error_string(void) { return g_err; }

int awq_check_device_error(void* stream) {
  // every stream's kernels report into the same per-device words
  AWQ_CUDA_TRY(cudaDeviceSynchronize());
  unsigned flags = 0;
  AWQ_TRY(read_clear_gemm_error(static_cast<cudaStream_t>(stream), &flags));
  unsigned narrow = 0;
  AWQ_TRY(read_clear_narrow_error(static_cast<cudaStream_t>(stream), &narrow));
  flags |= narrow << 8;
  unsigned gemv = 0;
  AWQ_TRY(read_clear_gemv_error(static_cast<cudaStream_t>(stream), &gemv));
  flags |= gemv << 16;
  if (flags) {
    set_error("a tensor-core matmul kernel gave up on a bounded wait (flags 0x%x)", flags);
    return AWQ_ERR_DEVICE;
  }
  return AWQ_OK;
}

size_t awq_absmean_workspace_size(int64_t T, int32_t K) {
  if (T <= 0 || K <= 0) return 0;
  return absmean_workspace_size(T, K);
}

int awq_absmean(const uint16_t* X, int64_t T, int32_t K, float* a, void* workspace,
                size_t ws_bytes, void* stream) {
  NvtxRange range("awq_absmean");
  if (T <= 0 || K <= 0 || K % kGroup != 0) {
    set_error("awq_absmean: T = %lld must be >= 1 and K = %d a positive multiple of 128",
              (long long)T, K);
    return AWQ_ERR_SHAPE;
  }
  AWQ_TRY(check_ptr(X, "X"));
  AWQ_TRY(check_ptr(a, "a"));
  if (!workspace || !aligned16(workspace) || ws_bytes < absmean_workspace_size(T, K)) {
    set_error("awq_absmean: workspace must be 16-B aligned and >= %zu bytes",
              absmean_workspace_size(T, K));
    return AWQ_ERR_WORKSPACE;
  }
  return launch_absmean(reinterpret_cast<const __half*>(X), T, K, a, workspace,
                        static_cast<cudaStream_t>(stream));
}

int awq_channel_scales(const float* a, int32_t K, double alpha, float* s_c, float* inv_s,
                       void* stream) {
  NvtxRange range("awq_channel_scales");
  if (K <= 0 || K % kGroup != 0) {
    set_error("awq_channel_scales: K = %d must be a positive multiple of 128", K);
    return AWQ_ERR_SHAPE;
  }
  if (!(alpha >= 0.0 && alpha < 1.0)) {
    set_error("awq_channel_scales: alpha = %g must lie in [0, 1)", alpha);
    return AWQ_ERR_SHAPE;
  }
  AWQ_TRY(check_ptr(a, "a"));
  AWQ_TRY(check_ptr(s_c, "s_c"));
  AWQ_TRY(check_ptr(inv_s, "inv_s"));
  return launch_channel_scales(a, K, alpha, s_c, inv_s, static_cast<cudaStream_t>(stream));
}

int awq_pack(const uint16_t* W, const float* s_c, int32_t N, int32_t K, const awq_config* cfg,
             uint32_t* qweight, uint16_t* scales, uint32_t* zeros, void* stream) {
  NvtxRange range("awq_pack");
  AWQ_TRY(check_cfg(cfg));
  AWQ_TRY(check_kn(N, K));
  AWQ_TRY(check_ptr(W, "W"));
  AWQ_TRY(check_opt_ptr(s_c, "s_c"));
  AWQ_TRY(check_ptr(qweight, "qweight"));
  AWQ_TRY(check_ptr(scales, "scales"));
  AWQ_TRY(check_ptr(zeros, "zeros"));
  const awq_config c = cfg ? *cfg : awq_default_config();
  AWQ_TRY(launch_pack(reinterpret_cast<const __half*>(W), s_c, N, K, qweight,
                      reinterpret_cast<__half*>(scales), zeros, static_cast<cudaStream_t>(stream),
                      c.w_bit, c.group, c.zero_point != 0));
  return launch_stream_fence(static_cast<cudaStream_t>(stream));
}

int awq_gemv_ex(const awq_config* cfg, const uint16_t* X, int32_t M, const uint32_t* qweight,
                const uint16_t* scales, const uint32_t* zeros, const float* inv_s, int32_t N,
                int32_t K, uint16_t* Y, void* stream) {
  NvtxRange range("awq_gemv_ex");
  AWQ_TRY(check_cfg(cfg));
  const awq_config c = cfg ? *cfg : awq_default_config();
  AWQ_TRY(check_kn(N, K));
  if (M < 1 || M > 8) {
    set_error("awq_gemv: M = %d must be in [1, 8]", M);
    return AWQ_ERR_SHAPE;
  }
  AWQ_TRY(check_ptr(X, "X"));
  AWQ_TRY(check_ptr(qweight, "qweight"));
  AWQ_TRY(check_ptr(scales, "scales"));
  AWQ_TRY(check_ptr(zeros, "zeros"));
  AWQ_TRY(check_opt_ptr(inv_s, "inv_s"));
  AWQ_TRY(check_ptr(Y, "Y"));
  return launch_gemv(reinterpret_cast<const __half*>(X), M, qweight,
                     reinterpret_cast<const __half*>(scales), zeros, inv_s, N, K,
                     reinterpret_cast<__half*>(Y), static_cast<cudaStream_t>(stream), false,
                     c.w_bit, c.group);
}

int awq_gemv(const uint16_t* X, int32_t M, const uint32_t* qweight, const uint16_t* scales,
             const uint32_t* zeros, const float* inv_s, int32_t N, int32_t K, uint16_t* Y,
             void* stream) {
  return awq_gemv_ex(nullptr, X, M, qweight, scales, zeros, inv_s, N, K, Y, stream);
}

int awq_gemv_silu_mul(const uint16_t* X, int32_t M, const uint32_t* qweight,
                      const uint16_t* scales, const uint32_t* zeros, const float* inv_s,
                      int32_t I, int32_t K, uint16_t* Y, void* stream) {
  NvtxRange range("awq_gemv_silu_mul");
  if (I <= 0 || I % 4 != 0) {
    set_error("awq_gemv_silu_mul: I = %d must be a positive multiple of 4", I);
    return AWQ_ERR_SHAPE;
  }
  AWQ_TRY(check_kn(2 * I, K));
  if (M < 1 || M > 8) {
    set_error("awq_gemv_silu_mul: M = %d must be in [1, 8]", M);
    return AWQ_ERR_SHAPE;
  }
  AWQ_TRY(check_ptr(X, "X"));
  AWQ_TRY(check_ptr(qweight, "qweight"));
  AWQ_TRY(check_ptr(scales, "scales"));
  AWQ_TRY(check_ptr(zeros, "zeros"));
  AWQ_TRY(check_opt_ptr(inv_s, "inv_s"));
  AWQ_TRY(check_ptr(Y, "Y"));
  return launch_gemv(reinterpret_cast<const __half*>(X), M, qweight,
                     reinterpret_cast<const __half*>(scales), zeros, inv_s, 2 * I, K,
                     reinterpret_cast<__half*>(Y), static_cast<cudaStream_t>(stream), true);
}

int awq_fold_inv_scales(const uint16_t* W, int64_t rows, int64_t cols, const float* inv_s,
                        uint16_t* out, void* stream) {
  NvtxRange range("awq_fold_inv_scales");
  if (rows < 1 || cols < 1) {
    set_error("awq_fold_inv_scales: rows = %lld and cols = %lld must be >= 1",
              static_cast<long long>(rows), static_cast<long long>(cols));
    return AWQ_ERR_SHAPE;
  }
  AWQ_TRY(check_ptr(W, "W"));
  AWQ_TRY(check_ptr(inv_s, "inv_s"));
  AWQ_TRY(check_ptr(out, "out"));
  return launch_fold_inv_scales(reinterpret_cast<const __half*>(W), rows, cols, inv_s,
                                reinterpret_cast<__half*>(out), static_cast<cudaStream_t>(stream));
}

namespace {
size_t xt_bytes(int32_t M, int32_t K) {
  return ((static_cast<size_t>(M) * K * 2 + 255) / 256) * 256;
}
}  // namespace

size_t awq_clip_search_workspace_size(int64_t T, int32_t K, const awq_config* cfg) {
  const awq_config c = cfg ? *cfg : awq_default_config();
  if (T <= 0 || K <= 0 || (c.group != 128 && c.group != 64 && c.group != 32) ||
      K % c.group != 0)
    return 0;
  return clip_workspace_size(T, K, c.group);
}

int awq_clip_search(const uint16_t* X_cal, int64_t T, const uint16_t* W, int32_t N, int32_t K,
                    const float* s_c, const float* inv_s, const awq_config* cfg, int32_t n_clip,
                    void* workspace, size_t ws_bytes, uint8_t* clip_idx, float* err_out,
                    void* stream) {
  NvtxRange range("awq_clip_search");
  AWQ_TRY(check_cfg(cfg));
  const awq_config c = cfg ? *cfg : awq_default_config();
  AWQ_TRY(check_kn(N, K));
  if (T < 1) {
    set_error("awq_clip_search: T = %lld must be >= 1", static_cast<long long>(T));
    return AWQ_ERR_SHAPE;
  }
  if (n_clip < 1 || n_clip > 200) {
    set_error("awq_clip_search: n_clip = %d must be in [1, 200]", n_clip);
    return AWQ_ERR_SHAPE;
  }
  AWQ_TRY(check_ptr(X_cal, "X_cal"));
  AWQ_TRY(check_ptr(W, "W"));
  AWQ_TRY(check_opt_ptr(s_c, "s_c"));
  AWQ_TRY(check_opt_ptr(inv_s, "inv_s"));
  AWQ_TRY(check_ptr(clip_idx, "clip_idx"));
  AWQ_TRY(check_opt_ptr(err_out, "err_out"));
  if (!workspace || !aligned16(workspace) ||
      ws_bytes < awq_clip_search_workspace_size(T, K, cfg)) {
    set_error("awq_clip_search: workspace must be 16-B aligned and >= %zu bytes",
              awq_clip_search_workspace_size(T, K, cfg));
    return AWQ_ERR_WORKSPACE;
  }
  return launch_clip_search(reinterpret_cast<const __half*>(X_cal), T,
                            reinterpret_cast<const __half*>(W), N, K, s_c, inv_s, c.w_bit,
                            c.group, c.zero_point != 0, n_clip, workspace, clip_idx, err_out,
                            static_cast<cudaStream_t>(stream));
}

int awq_pack_clipped(const uint16_t* W, const float* s_c, int32_t N, int32_t K,
                     const awq_config* cfg, const uint8_t* clip_idx, int32_t n_clip,
                     uint32_t* qweight, uint16_t* scales, uint32_t* zeros, void* stream) {
  NvtxRange range("awq_pack_clipped");
  AWQ_TRY(check_cfg(cfg));
  AWQ_TRY(check_kn(N, K));
  if (n_clip < 1 || n_clip > 200) {
    set_error("awq_pack_clipped: n_clip = %d must be in [1, 200]", n_clip);
    return AWQ_ERR_SHAPE;
  }
  AWQ_TRY(check_ptr(W, "W"));
  AWQ_TRY(check_opt_ptr(s_c, "s_c"));
  AWQ_TRY(check_ptr(clip_idx, "clip_idx"));
  AWQ_TRY(check_ptr(qweight, "qweight"));
  AWQ_TRY(check_ptr(scales, "scales"));
  AWQ_TRY(check_ptr(zeros, "zeros"));
  const awq_config c = cfg ? *cfg : awq_default_config();
  AWQ_TRY(launch_pack(reinterpret_cast<const __half*>(W), s_c, N, K, qweight,
                      reinterpret_cast<__half*>(scales), zeros, static_cast<cudaStream_t>(stream),
                      c.w_bit, c.group, c.zero_point != 0, clip_idx, n_clip));
  return launch_stream_fence(static_cast<cudaStream_t>(stream));
}

size_t awq_gemm_workspace_size(int32_t M, int32_t N, int32_t K) {
  if (M <= 0 || K <= 0 || N <= 0 || K % kGroup != 0) return 0;
  return xt_bytes(M, K) + gemm_partial_bytes(M, N, K);
}

namespace {

int gemm_common(int mode, const awq_config* cfg, const uint16_t* X, int32_t M,
                const uint32_t* qweight, const uint16_t* scales, const uint32_t* zeros,
                const float* inv_s, int32_t N, int32_t K, uint16_t* Y, int32_t ldy,
                void* workspace, size_t ws_bytes, void* stream) {
  NvtxRange range(mode == kGemmSiluF16 ? "awq_gemm_silu_mul" : "awq_gemm");
  AWQ_TRY(check_cfg(cfg));
  const awq_config c = cfg ? *cfg : awq_default_config();
  AWQ_TRY(check_kn(N, K));
  if (M < 1) {
    set_error("awq_gemm: M = %d must be >= 1", M);
    return AWQ_ERR_SHAPE;
  }
  AWQ_TRY(check_ptr(X, "X"));
  AWQ_TRY(check_ptr(qweight, "qweight"));
  AWQ_TRY(check_ptr(scales, "scales"));
  AWQ_TRY(check_ptr(zeros, "zeros"));
  AWQ_TRY(check_opt_ptr(inv_s, "inv_s"));
  AWQ_TRY(check_ptr(Y, "Y"));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (inv_s && (!workspace || !aligned16(workspace) || ws_bytes < xt_bytes(M, K))) {
    set_error("awq_gemm: workspace must be 16-B aligned and >= %zu bytes",
              awq_gemm_workspace_size(M, N, K));
    return AWQ_ERR_WORKSPACE;
  }
  // up to 8 tokens of the default format: the decode matmul (warp-level MMA,
  // weights streamed by TMA) when it runs without a K split or with K halved
  // over a cluster of two; it scales the activations itself, so the
  // workspace is not used
  if (mode == kGemmOutF16 && gemv_mma_eligible(M, K, c.w_bit, c.group, false)) {
    const MmaGemvPlan p = plan_gemv_mma(M, N, K, sm_count());
    if (p.depth > 0 && p.nsplit <= 2)
      return launch_gemv_mma_plan(p, reinterpret_cast<const __half*>(X), M, qweight,
                                  reinterpret_cast<const __half*>(scales), zeros, inv_s, N, K,
                                  reinterpret_cast<__half*>(Y), st);
  }
  const __half* xt = reinterpret_cast<const __half*>(X);
  // workspace: X~ first (when inv_s is given), then the split-K partial sums
  // if the rest of the workspace holds them
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  size_t rest = ws_bytes;
  if (inv_s) {
    if (!workspace || !aligned16(workspace) || ws_bytes < xt_bytes(M, K)) {
      set_error("awq_gemm: workspace must be 16-B aligned and >= %zu bytes",
                awq_gemm_workspace_size(M, N, K));
      return AWQ_ERR_WORKSPACE;
    }
    __half* w = reinterpret_cast<__half*>(ws);
    AWQ_TRY(launch_prescale(xt, inv_s, M, K, w, st, c.w_bit));
    xt = w;
    ws += xt_bytes(M, K);
    rest -= xt_bytes(M, K);
  }
  float* part = (ws && aligned16(ws)) ? reinterpret_cast<float*>(ws) : nullptr;
  return launch_gemm(mode, xt, inv_s != nullptr, M, qweight,
                     reinterpret_cast<const __half*>(scales), zeros, nullptr, N, K, Y, ldy,
                     nullptr, 0, st, c.w_bit, c.group, part, part ? rest : 0);
}

}  // namespace

int awq_gemm(const uint16_t* X, int32_t M, const uint32_t* qweight, const uint16_t* scales,
             const uint32_t* zeros, const float* inv_s, int32_t N, int32_t K, uint16_t* Y,
             void* workspace, size_t ws_bytes, void* stream) {
  return gemm_common(kGemmOutF16, nullptr, X, M, qweight, scales, zeros, inv_s, N, K, Y, N,
                     workspace, ws_bytes, stream);
}

int awq_gemm_ex(const awq_config* cfg, const uint16_t* X, int32_t M, const uint32_t* qweight,
                const uint16_t* scales, const uint32_t* zeros, const float* inv_s, int32_t N,
                int32_t K, uint16_t* Y, void* workspace, size_t ws_bytes, void* stream) {
  return gemm_common(kGemmOutF16, cfg, X, M, qweight, scales, zeros, inv_s, N, K, Y, N,
                     workspace, ws_bytes, stream);
}

int awq_gemm_silu_mul(const uint16_t* X, int32_t M, const uint32_t* qweight,
                      const uint16_t* scales, const uint32_t* zeros, const float* inv_s,
                      int32_t I, int32_t K, uint16_t* Y, void* workspace, size_t ws_bytes,
                      void* stream) {
  if (I <= 0 || I % 4 != 0) {
    set_error("awq_gemm_silu_mul: I = %d must be a positive multiple of 4", I);
    return AWQ_ERR_SHAPE;
  }
  return gemm_common(kGemmSiluF16, nullptr, X, M, qweight, scales, zeros, inv_s, 2 * I, K, Y, I,
                     workspace, ws_bytes, stream);
}

int awq_debug_stall(int32_t which, int64_t wait_limit_ns) {
  if (which < 0 || which > 3) {
    set_error("awq_debug_stall: which = %d must be a combination of 1 and 2", which);
    return AWQ_ERR_SHAPE;
  }
  if (wait_limit_ns < 1000 || wait_limit_ns > 10000000000ll) {
    set_error("awq_debug_stall: wait_limit_ns = %lld must be in [1e3, 1e10]",
              static_cast<long long>(wait_limit_ns));
    return AWQ_ERR_SHAPE;
  }
  AWQ_TRY(set_gemv_stall(which & 1, static_cast<uint64_t>(wait_limit_ns)));
  return set_gemm_stall(which & 2, static_cast<uint64_t>(wait_limit_ns));
}

int awq_measure_stream_read(const void* buf, size_t bytes, int32_t read_first, uint32_t* out,
                            void* stream) {
  NvtxRange range("awq_measure_stream_read");
  if (bytes == 0 || bytes % 16 != 0) {
    set_error("awq_measure_stream_read: bytes = %zu must be a positive multiple of 16", bytes);
    return AWQ_ERR_SHAPE;
  }
  AWQ_TRY(check_ptr(buf, "buf"));
  AWQ_TRY(check_ptr(out, "out"));
  return launch_stream_read(buf, bytes, read_first, out, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
