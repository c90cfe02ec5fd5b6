// Row-wise kernels between the projections: embedding gather + RMSNorm, the
// QKV epilogue (split-K reduction, RoPE, paged KV write), residual add +
// RMSNorm, and the SwiGLU epilogue.  All are memory/latency bound and touch
// only the B*W rows of the round (linear layers act on the flattened rows:
// Lecture 6 "Optimizing Autoregressive Decode", section 4.2).
#include "common.cuh"
#include "launch.cuh"

namespace spec {

namespace {

template <int NT>
__device__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x < 32) {
    t = threadIdx.x < NT / 32 ? red[threadIdx.x] : 0.f;
    t = warp_sum(t);
    if (threadIdx.x == 0) red[32] = t;
  }
  __syncthreads();
  t = red[32];
  __syncthreads();
  return t;
}

constexpr int kRowThreads = 256;

// resid[m] = E[tok[m]] (fp32); xn[m] = bf16(rmsnorm(resid[m]) * g)
__global__ void __launch_bounds__(kRowThreads) embed_norm_kernel(const int32_t* tok, const __nv_bfloat16* embed,
                                                                 const float* gain, int d, int vocab, float eps,
                                                                 float* resid, __nv_bfloat16* xn, int* status) {
  __shared__ float red[33];
  pdl_wait();
  pdl_launch_dependents();
  const int m = blockIdx.x;
  int t = tok[m];
  if (t < 0 || t >= vocab) {
    set_status(status, SPEC_ERR_INVALID_ARG);
    t = 0;
  }
  const __nv_bfloat16* e = embed + (long long)t * d;
  float* r = resid + (long long)m * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += kRowThreads) {
    const float v = __bfloat162float(e[i]);
    r[i] = v;
    ss += v * v;
  }
  ss = block_sum<kRowThreads>(ss, red);
  const float inv = rsqrtf(ss / d + eps);
  for (int i = threadIdx.x; i < d; i += kRowThreads) xn[(long long)m * d + i] = __float2bfloat16(r[i] * inv * gain[i]);
}

// resid[m] += sum_s part[s][m]; xn[m] = bf16(rmsnorm(resid[m]) * g)
__global__ void __launch_bounds__(kRowThreads) resid_norm_kernel(const float* part, int splits, long long split_stride,
                                                                 int d, const float* gain, float eps, float* resid,
                                                                 __nv_bfloat16* xn) {
  __shared__ float red[33];
  pdl_wait();
  pdl_launch_dependents();
  const int m = blockIdx.x;
  float* r = resid + (long long)m * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += kRowThreads) {
    float v = r[i];
    for (int s = 0; s < splits; ++s) v += part[s * split_stride + (long long)m * d + i];
    r[i] = v;
    ss += v * v;
  }
  ss = block_sum<kRowThreads>(ss, red);
  const float inv = rsqrtf(ss / d + eps);
  for (int i = threadIdx.x; i < d; i += kRowThreads) xn[(long long)m * d + i] = __float2bfloat16(r[i] * inv * gain[i]);
}

// One thread per (row, head, rotation pair).  Column layout of the fused QKV
// output: q heads, then k heads, then v heads, each head_dim wide.
// RoPE (half-split): (a, b) -> (a cos - b sin, a sin + b cos) with the angle
// table of the row's position.
__global__ void __launch_bounds__(kRowThreads) qkv_epilogue_kernel(
    const float* part, int splits, long long split_stride, int n_heads, int n_kv, int hd, const int32_t* row_pos,
    const int32_t* row_slot, const float* rope_cos, const float* rope_sin, __nv_bfloat16* q_out,
    __nv_bfloat16* kpool, __nv_bfloat16* vpool) {
  pdl_wait();
  pdl_launch_dependents();
  const int m = blockIdx.y;
  const int half = hd >> 1;
  const int n_pairs = (n_heads + 2 * n_kv) * half;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_pairs) return;
  const int head = idx / half;  // 0..n_heads+2*n_kv-1
  const int i = idx - head * half;
  const int N = (n_heads + 2 * n_kv) * hd;
  const long long base = (long long)m * N + (long long)head * hd;
  float a = 0.f, b = 0.f;
  for (int s = 0; s < splits; ++s) {
    a += part[s * split_stride + base + i];
    b += part[s * split_stride + base + i + half];
  }
  const int pos = row_pos[m];
  if (head < n_heads + n_kv) {  // q or k: rotate
    const float c = rope_cos[(long long)pos * half + i];
    const float sn = rope_sin[(long long)pos * half + i];
    const float ra = a * c - b * sn;
    const float rb = a * sn + b * c;
    a = ra;
    b = rb;
  }
  if (head < n_heads) {
    __nv_bfloat16* q = q_out + (long long)m * n_heads * hd + (long long)head * hd;
    q[i] = __float2bfloat16(a);
    q[i + half] = __float2bfloat16(b);
    return;
  }
  const int slot = row_slot[m];
  if (slot < 0) return;  // the round failed to get a page for this row
  const int page = slot / kPage, off = slot % kPage;
  const bool is_k = head < n_heads + n_kv;
  const int kvh = is_k ? head - n_heads : head - n_heads - n_kv;
  __nv_bfloat16* dst = (is_k ? kpool : vpool) + (((long long)page * n_kv + kvh) * kPage + off) * hd;
  dst[i] = __float2bfloat16(a);
  dst[i + half] = __float2bfloat16(b);
}

// act[m][f] = bf16(silu(gate) * up); gate/up rows are interleaved in 64-row
// blocks: physical row 128*j + r is gate row 64*j + r (r < 64) or up row
// 64*j + r - 64 (r >= 64).
__global__ void __launch_bounds__(kRowThreads) swiglu_kernel(const float* part, int splits, long long split_stride,
                                                             int ffn, __nv_bfloat16* act) {
  pdl_wait();
  pdl_launch_dependents();
  const int m = blockIdx.y;
  const int f = blockIdx.x * blockDim.x + threadIdx.x;
  if (f >= ffn) return;
  const long long N = 2LL * ffn;
  const long long pg = (long long)(f >> 6) * 128 + (f & 63);
  float g = 0.f, u = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float* ps = part + s * split_stride + (long long)m * N;
    g += ps[pg];
    u += ps[pg + 64];
  }
  const float silu = g / (1.f + expf(-g));
  act[(long long)m * ffn + f] = __float2bfloat16(silu * u);
}

}  // namespace

cudaError_t launch_embed_norm(const int32_t* tok, int M, const __nv_bfloat16* embed, const float* gain, int d,
                              int vocab, float eps, float* resid, __nv_bfloat16* xn, int* status, cudaStream_t st) {
  return launch_k(embed_norm_kernel, dim3(M), dim3(kRowThreads), 0, st, tok, embed, gain, d, vocab, eps, resid, xn,
                  status);
}

cudaError_t launch_resid_norm(const float* part, int splits, long long split_stride, int M, int d, const float* gain,
                              float eps, float* resid, __nv_bfloat16* xn, cudaStream_t st) {
  return launch_k(resid_norm_kernel, dim3(M), dim3(kRowThreads), 0, st, part, splits, split_stride, d, gain, eps,
                  resid, xn);
}

cudaError_t launch_qkv_epilogue(const float* part, int splits, long long split_stride, int M, int n_heads, int n_kv,
                                int hd, const int32_t* row_pos, const int32_t* row_slot, const float* rope_cos,
                                const float* rope_sin, __nv_bfloat16* q_out, __nv_bfloat16* kpool_layer,
                                __nv_bfloat16* vpool_layer, cudaStream_t st) {
  const int n_pairs = (n_heads + 2 * n_kv) * (hd / 2);
  dim3 grid((n_pairs + kRowThreads - 1) / kRowThreads, M);
  return launch_k(qkv_epilogue_kernel, grid, dim3(kRowThreads), 0, st, part, splits, split_stride, n_heads, n_kv, hd,
                  row_pos, row_slot, rope_cos, rope_sin, q_out, kpool_layer, vpool_layer);
}

cudaError_t launch_swiglu(const float* part, int splits, long long split_stride, int M, int ffn, __nv_bfloat16* act,
                          cudaStream_t st) {
  dim3 grid((ffn + kRowThreads - 1) / kRowThreads, M);
  return launch_k(swiglu_kernel, grid, dim3(kRowThreads), 0, st, part, splits, split_stride, ffn, act);
}

}  // namespace spec
