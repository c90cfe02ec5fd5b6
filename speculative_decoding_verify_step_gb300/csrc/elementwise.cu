// Embedding gather that starts the residual stream of a round (linear layers
// act on the flattened B*W rows: Lecture 6 "Optimizing Autoregressive Decode",
// section 4.2).  It also prepares the first RMSNorm in the folded form the
// projections consume: X' = bf16(r * g) and, per 128-column tile, sum r^2 (the
// QKV projection scales its output rows by rsqrt(sum r^2 / d + eps)).
#include "common.cuh"
#include "launch.cuh"

namespace spec {

namespace {

constexpr int kTileCols = 128;

// grid (M, d / 128), 128 threads: one column per thread, one tile per block.
__global__ void __launch_bounds__(kTileCols) embed_kernel(const int32_t* tok, const __nv_bfloat16* embed,
                                                          const float* gain, int d, int vocab, float* resid,
                                                          __nv_bfloat16* xn, float* ssq_out, int ssq_stride,
                                                          int* status) {
  __shared__ float red[kTileCols / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int m = blockIdx.x;
  const int col = blockIdx.y * kTileCols + threadIdx.x;
  int t = tok[m];
  if (t < 0 || t >= vocab) {
    if (threadIdx.x == 0 && blockIdx.y == 0) set_status(status, SPEC_ERR_INVALID_ARG);
    t = 0;
  }
  const float v = __bfloat162float(embed[(long long)t * d + col]);
  resid[(long long)m * d + col] = v;
  xn[(long long)m * d + col] = __float2bfloat16(v * gain[col]);
  float ss = warp_sum(v * v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < kTileCols / 32; ++w) s += red[w];
    ssq_out[(long long)blockIdx.y * ssq_stride + m] = s;
  }
}

}  // namespace

cudaError_t launch_embed(const int32_t* tok, int M, const __nv_bfloat16* embed, const float* gain, int d, int vocab,
                         float* resid, __nv_bfloat16* xn, float* ssq_out, int ssq_stride, int* status,
                         cudaStream_t st) {
  return launch_k(embed_kernel, dim3(M, d / kTileCols), dim3(kTileCols), 0, st, tok, embed, gain, d, vocab, resid,
                  xn, ssq_out, ssq_stride, status);
}

}  // namespace spec
