// Embedding gather that starts the residual stream of a round (linear layers
// act on the flattened B*W rows: Lecture 6 "Optimizing Autoregressive Decode",
// section 4.2).  It also prepares the first RMSNorm in the folded form the
// projections consume: X' = fp16(r * g) and, per 128-column tile, sum r^2 (the
// QKV projection scales its output rows by rsqrt(sum r^2 / d + eps)).
#include "common.cuh"
#include "launch.cuh"

namespace spec {

namespace {

constexpr int kTileCols = 128;

// grid (M, d / 128), 128 threads: one column per thread, one tile per block.
__global__ void __launch_bounds__(kTileCols) embed_kernel(const int32_t* tok, const __nv_bfloat16* embed,
                                                          const float* gain, int d, int vocab, float* resid,
                                                          act_t* xn, float* ssq_out, int ssq_stride,
                                                          int* status) {
  __shared__ float red[kTileCols / 32];
  // The first projection may start streaming its weights now: it reads nothing of
  // this kernel's (or the round preparation's) output before its own dependency
  // wait, which returns once this grid, and so the preparation before it, is done.
  pdl_launch_dependents();
  pdl_wait();
  const int m = blockIdx.x;
  const int col = blockIdx.y * kTileCols + threadIdx.x;
  int t = tok[m];
  if (t < 0 || t >= vocab) {
    if (threadIdx.x == 0 && blockIdx.y == 0) set_status(status, SPEC_ERR_INVALID_ARG);
    t = 0;
  }
  const float v = __bfloat162float(embed[(long long)t * d + col]);
  resid[(long long)m * d + col] = v;
  xn[(long long)m * d + col] = to_act(v * gain[col]);
  float ss = warp_sum(v * v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < kTileCols / 32; ++w) s += red[w];
    ssq_out[(long long)blockIdx.y * ssq_stride + m] = s;
  }
}

// In-place re-encoding of bf16 weight rows as fp16 times a power of two.  Row i of
// the list is physical row (i / block) * block_stride + row0 + i % block.  With
// the row's largest magnitude in [2^(E-1), 2^E) the row is multiplied by 2^e,
// e = 15 - E, so its largest value lands in [2^14, 2^15): every bf16 value of the
// row that is at most 2^32 times smaller than the row maximum is represented
// exactly (fp16 normals and the upper subnormals hold the 8 significant bits).
// rscale[row] = 2^-e undoes the scaling in the projection epilogue.
__global__ void __launch_bounds__(256) encode_rows_kernel(uint16_t* w, int K, int block, int block_stride, int row0,
                                                          float* rscale) {
  __shared__ float red[8];
  const int i = blockIdx.x;
  const long long row = (long long)(i / block) * block_stride + row0 + i % block;
  uint16_t* r = w + row * K;
  float mx = 0.f;
  for (int k = threadIdx.x; k < K; k += 256) mx = fmaxf(mx, fabsf(__uint_as_float((uint32_t)r[k] << 16)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = red[0];
  for (int j = 1; j < 8; ++j) mx = fmaxf(mx, red[j]);
  int E = 0;
  if (mx > 0.f) frexpf(mx, &E);
  const int e = mx > 0.f ? 15 - E : 0;
  const float s = ldexpf(1.f, e);
  for (int k = threadIdx.x; k < K; k += 256) {
    const float v = __uint_as_float((uint32_t)r[k] << 16) * s;
    r[k] = __half_as_ushort(__float2half_rn(v));
  }
  if (threadIdx.x == 0) rscale[row] = ldexpf(1.f, -e);
}

}  // namespace

cudaError_t launch_encode_rows(uint16_t* w, int K, int n_rows, int block, int block_stride, int row0, float* rscale,
                               cudaStream_t st) {
  encode_rows_kernel<<<n_rows, 256, 0, st>>>(w, K, block, block_stride, row0, rscale);
  return cudaGetLastError();
}

cudaError_t launch_embed(const int32_t* tok, int M, const __nv_bfloat16* embed, const float* gain, int d, int vocab,
                         float* resid, act_t* xn, float* ssq_out, int ssq_stride, int* status,
                         cudaStream_t st) {
  return launch_k(embed_kernel, dim3(M, d / kTileCols), dim3(kTileCols), 0, st, tok, embed, gain, d, vocab, resid,
                  xn, ssq_out, ssq_stride, status);
}

}  // namespace spec
