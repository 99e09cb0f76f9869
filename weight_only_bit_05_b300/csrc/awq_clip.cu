// Per-group weight-clipping search.
//
// "AWQ量化实战：无需重训，把大模型压进4bit显存" §5.1 names a clipping parameter
// (clip_steps) and nothing more.  The library's reading: after the scale
// search, each group's range of scaled weights may shrink to [r min, r max],
// r_i = 1 - 0.5 i / n (i = 0 .. n-1); the group is quantized from the shrunk
// range, and the ratio with the smallest output error on the calibration
// tokens is kept (ties: the least clipping).  The error of group g of row n
// is d^T H_g d with d = w^ - w' (the dequantized minus the scaled weights)
// and H_g = X~_g^T X~_g the Gram matrix of the group's scaled activations.
//
//  * gram_partial_kernel: one CTA per (group, token chunk) accumulates the
//    GS x GS outer products of its tokens in fp32 registers (x~ = fp32(x) *
//    inv_s, as the layer computes it); gram_reduce_kernel adds the chunks in
//    order (deterministic);
//  * clip_search_kernel: one CTA per (group, block of rows) holds H_g in
//    shared memory; a warp takes a row, each lane GS/32 of its weights.  For
//    four candidate ratios at a time the lanes quantize their weights exactly
//    as the pack kernel does, write d to shared memory, and form H_g d with
//    each 16-byte load of H_g serving the four candidates.
#include "awq_internal.h"

namespace awq {
namespace {

constexpr int kTokChunk = 1024;   // tokens per Gram partial
constexpr int kMaxChunks = 16;
constexpr int kRowsPerCta = 32;   // rows of a clip-search CTA (8 warps x 4)
constexpr int kCand = 4;          // candidates per pass

__device__ __forceinline__ float clip_ratio_dev(int i, int n) {
  return __double2float_rn(__dsub_rn(1.0, __ddiv_rn(__dmul_rn(0.5, static_cast<double>(i)),
                                                    static_cast<double>(n))));
}

template <int GS>
__global__ void __launch_bounds__(256)
    gram_partial_kernel(const __half* __restrict__ X, int64_t T, int K,
                        const float* __restrict__ inv_s, int64_t tok_per_chunk,
                        float* __restrict__ part) {
  constexpr int TILE = GS / 16;            // a thread's TILE x TILE block of H
  constexpr int kTok = 32;                 // tokens staged per step
  __shared__ float xs[kTok][GS];
  const int g = blockIdx.x, tc = blockIdx.y;
  const int ti = threadIdx.x / 16, tj = threadIdx.x % 16;
  const int64_t t0 = tc * tok_per_chunk;
  const int64_t t1 = t0 + tok_per_chunk < T ? t0 + tok_per_chunk : T;
  float acc[TILE][TILE];
#pragma unroll
  for (int a = 0; a < TILE; ++a)
#pragma unroll
    for (int b = 0; b < TILE; ++b) acc[a][b] = 0.f;
  for (int64_t tb = t0; tb < t1; tb += kTok) {
    __syncthreads();
    for (int e = threadIdx.x; e < kTok * GS; e += 256) {
      const int tt = e / GS, k = e - tt * GS;
      const int64_t t = tb + tt;
      float v = 0.f;
      if (t < t1) {
        v = __half2float(X[t * K + static_cast<int64_t>(g) * GS + k]);
        if (inv_s) v = __fmul_rn(v, inv_s[g * GS + k]);
      }
      xs[tt][k] = v;
    }
    __syncthreads();
#pragma unroll 4
    for (int tt = 0; tt < kTok; ++tt) {
      float a[TILE], b[TILE];
#pragma unroll
      for (int i = 0; i < TILE; ++i) {
        a[i] = xs[tt][ti * TILE + i];
        b[i] = xs[tt][tj * TILE + i];
      }
#pragma unroll
      for (int i = 0; i < TILE; ++i)
#pragma unroll
        for (int j = 0; j < TILE; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
  }
  float* dst = part + (static_cast<size_t>(g) * gridDim.y + tc) * GS * GS;
#pragma unroll
  for (int i = 0; i < TILE; ++i)
#pragma unroll
    for (int j = 0; j < TILE; ++j) dst[(ti * TILE + i) * GS + tj * TILE + j] = acc[i][j];
}

__global__ void gram_reduce_kernel(const float* __restrict__ part, int chunks, int64_t per_group,
                                   int64_t total, float* __restrict__ H) {
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t g = e / per_group, i = e - g * per_group;
    const float* p = part + g * chunks * per_group + i;
    float v = p[0];
    for (int c = 1; c < chunks; ++c) v += p[c * per_group];
    H[e] = v;
  }
}

template <int BITS, int GS, bool ZP>
__global__ void __launch_bounds__(256)
    clip_search_kernel(const __half* __restrict__ W, int N, int K, const float* __restrict__ s_c,
                       const float* __restrict__ H, int n_clip, uint8_t* __restrict__ clip_idx,
                       float* __restrict__ err) {
  constexpr int C = GS / 32;               // weights of a lane
  constexpr int kQmax = (1 << BITS) - 1;
  constexpr int kHalf = 1 << (BITS - 1);
  extern __shared__ float smem_f[];
  float* Hs = smem_f;                                  // [GS][GS]
  float* dsm = Hs + GS * GS;                           // [8 warps][kCand][GS]
  const int g = blockIdx.x;
  const int G = K / GS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float4* Hg = reinterpret_cast<const float4*>(H + static_cast<size_t>(g) * GS * GS);
  for (int e = threadIdx.x; e < GS * GS / 4; e += 256) reinterpret_cast<float4*>(Hs)[e] = Hg[e];
  __syncthreads();
  float* dw = dsm + warp * kCand * GS;

  for (int rr = 0; rr < kRowsPerCta / 8; ++rr) {
    const int n = blockIdx.y * kRowsPerCta + warp * (kRowsPerCta / 8) + rr;
    if (n >= N) break;                                 // warp-uniform
    float w[C];
#pragma unroll
    for (int a = 0; a < C; ++a) {
      const int k = g * GS + lane * C + a;
      w[a] = __half2float(W[static_cast<size_t>(n) * K + k]);
      if (s_c) w[a] = __fmul_rn(w[a], s_c[k]);
    }
    float mn = w[0], mx = w[0];
#pragma unroll
    for (int a = 1; a < C; ++a) {
      mn = fminf(mn, w[a]);
      mx = fmaxf(mx, w[a]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    }
    const float amax = fmaxf(fabsf(mn), fabsf(mx));
    float best_e = 0.f;
    int best_i = 0;
    for (int i0 = 0; i0 < n_clip; i0 += kCand) {
      float d[kCand][C];
#pragma unroll
      for (int c = 0; c < kCand; ++c) {
        const int i = i0 + c < n_clip ? i0 + c : n_clip - 1;
        const float r = clip_ratio_dev(i, n_clip);
        // the pack kernel's step, zero point and codes for the shrunk range
        const float cmn = __fmul_rn(mn, r), cmx = __fmul_rn(mx, r), cam = __fmul_rn(amax, r);
        float s32 = ZP ? __fdiv_rn(__fsub_rn(cmx, cmn), static_cast<float>(kQmax))
                       : __fdiv_rn(cam, static_cast<float>(kHalf - 1));
        s32 = fminf(fmaxf(s32, 6.103515625e-05f), 65504.0f);
        const float s = __half2float(__float2half_rn(s32));
        const float z = ZP ? fminf(fmaxf(rintf(__fdiv_rn(-cmn, s)), 0.f), static_cast<float>(kQmax))
                           : static_cast<float>(kHalf);
#pragma unroll
        for (int a = 0; a < C; ++a) {
          const float rq = rintf(__fdiv_rn(w[a], s));
          const float q = ZP ? fminf(fmaxf(rq + z, 0.f), static_cast<float>(kQmax))
                             : fminf(fmaxf(rq, static_cast<float>(-kHalf)),
                                     static_cast<float>(kHalf - 1)) + static_cast<float>(kHalf);
          d[c][a] = __fsub_rn(__fmul_rn(q - z, s), w[a]);
          dw[c * GS + lane * C + a] = d[c][a];
        }
      }
      __syncwarp();
      // e_c = d_c^T H d_c; lane accumulates (H d_c) for its own C rows of H
      float hd[kCand][C];
#pragma unroll
      for (int c = 0; c < kCand; ++c)
#pragma unroll
        for (int a = 0; a < C; ++a) hd[c][a] = 0.f;
#pragma unroll 4
      for (int j = 0; j < GS; ++j) {
        float hv[C];
#pragma unroll
        for (int a = 0; a < C; ++a) hv[a] = Hs[j * GS + lane * C + a];   // H[j][k] = H[k][j]
#pragma unroll
        for (int c = 0; c < kCand; ++c) {
          const float dj = dw[c * GS + j];
#pragma unroll
          for (int a = 0; a < C; ++a) hd[c][a] = fmaf(hv[a], dj, hd[c][a]);
        }
      }
#pragma unroll
      for (int c = 0; c < kCand; ++c) {
        float e = 0.f;
#pragma unroll
        for (int a = 0; a < C; ++a) e = fmaf(d[c][a], hd[c][a], e);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) e += __shfl_xor_sync(0xffffffffu, e, off);
        const int i = i0 + c;
        if (i < n_clip) {
          if (err && lane == 0) err[(static_cast<size_t>(n) * G + g) * n_clip + i] = e;
          if (i == 0 || e < best_e) {
            best_e = e;
            best_i = i;
          }
        }
      }
      __syncwarp();
    }
    if (lane == 0) clip_idx[static_cast<size_t>(n) * G + g] = static_cast<uint8_t>(best_i);
  }
}

int chunks_for(int64_t T) {
  int64_t c = (T + kTokChunk - 1) / kTokChunk;
  return static_cast<int>(c < kMaxChunks ? (c < 1 ? 1 : c) : kMaxChunks);
}

template <int GS>
int launch_gram(const __half* X, int64_t T, int K, const float* inv_s, float* part, float* H,
                cudaStream_t st) {
  const int G = K / GS;
  const int chunks = chunks_for(T);
  const int64_t per = (T + chunks - 1) / chunks;
  gram_partial_kernel<GS><<<dim3(G, chunks), 256, 0, st>>>(X, T, K, inv_s, per, part);
  AWQ_CUDA_TRY_LAUNCH("gram_partial_kernel");
  const int64_t total = static_cast<int64_t>(G) * GS * GS;
  gram_reduce_kernel<<<static_cast<unsigned>((total + 255) / 256 < 4096 ? (total + 255) / 256
                                                                        : 4096),
                       256, 0, st>>>(part, chunks, static_cast<int64_t>(GS) * GS, total, H);
  AWQ_CUDA_TRY_LAUNCH("gram_reduce_kernel");
  return AWQ_OK;
}

template <int BITS, int GS, bool ZP>
int launch_search(const __half* W, int N, int K, const float* s_c, const float* H, int n_clip,
                  uint8_t* clip_idx, float* err, cudaStream_t st) {
  const size_t smem = (static_cast<size_t>(GS) * GS + 8 * kCand * GS) * sizeof(float);
  {
    const int rc = ensure_smem_attr(reinterpret_cast<const void*>(clip_search_kernel<BITS, GS, ZP>),
                                    static_cast<int>(smem));
    if (rc != AWQ_OK) return rc;
  }
  const dim3 grid(K / GS, (N + kRowsPerCta - 1) / kRowsPerCta);
  clip_search_kernel<BITS, GS, ZP><<<grid, 256, smem, st>>>(W, N, K, s_c, H, n_clip, clip_idx,
                                                            err);
  AWQ_CUDA_TRY_LAUNCH("clip_search_kernel");
  return AWQ_OK;
}

}  // namespace

size_t clip_workspace_size(int64_t T, int K, int group) {
  const int chunks = chunks_for(T);
  const size_t per = static_cast<size_t>(K / group) * group * group * sizeof(float);
  return ((per * (chunks + 1) + 255) / 256) * 256;
}

int launch_clip_search(const __half* X, int64_t T, const __half* W, int N, int K,
                       const float* s_c, const float* inv_s, int w_bit, int group,
                       bool zero_point, int n_clip, void* ws, uint8_t* clip_idx, float* err,
                       cudaStream_t st) {
  float* H = static_cast<float*>(ws);
  float* part = H + static_cast<size_t>(K / group) * group * group;
  int rc;
  if (group == 128) rc = launch_gram<128>(X, T, K, inv_s, part, H, st);
  else if (group == 64) rc = launch_gram<64>(X, T, K, inv_s, part, H, st);
  else rc = launch_gram<32>(X, T, K, inv_s, part, H, st);
  if (rc != AWQ_OK) return rc;
#define AWQ_CLIP_CASE(B, GS, ZP)                                                               \
  if (w_bit == B && group == GS && zero_point == ZP)                                           \
    return launch_search<B, GS, ZP>(W, N, K, s_c, H, n_clip, clip_idx, err, st);
  AWQ_CLIP_CASE(4, 128, true)
  AWQ_CLIP_CASE(4, 64, true)
  AWQ_CLIP_CASE(4, 32, true)
  AWQ_CLIP_CASE(4, 128, false)
  AWQ_CLIP_CASE(4, 64, false)
  AWQ_CLIP_CASE(4, 32, false)
  AWQ_CLIP_CASE(8, 128, true)
  AWQ_CLIP_CASE(8, 64, true)
  AWQ_CLIP_CASE(8, 32, true)
  AWQ_CLIP_CASE(8, 128, false)
  AWQ_CLIP_CASE(8, 64, false)
  AWQ_CLIP_CASE(8, 32, false)
#undef AWQ_CLIP_CASE
  set_error("awq_clip_search: unsupported configuration");
  return AWQ_ERR_UNSUPPORTED;
}

}  // namespace awq
