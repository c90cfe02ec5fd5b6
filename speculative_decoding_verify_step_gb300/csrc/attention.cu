// Paged attention for the verify window.
//
// One CTA per (sequence, kv head, KV split).  All gamma+1 query rows of the
// sequence and all query heads that share the kv head (grouped-query
// attention) sit in the same CTA, so every K/V page is loaded from HBM once for
// all of them (Lecture 6 "Optimizing Autoregressive Decode", section 9.2: the
// gamma+1 queries of one sequence share one KV read inside a fused kernel).
// Attention is per sequence against its own cache (section 4.2).
//
// Masking covers both window shapes: a window row j sees every cached slot
// < L and the window slots of its ancestors (bit i of anc[j]); a chain is the
// tree whose ancestors of j are 0..j (section 10.3: each tree node sees only
// its ancestors).
//
// K/V pages (64 tokens x head_dim bf16 per kv head) are streamed by TMA with
// the 128-byte swizzle into a 3-stage mbarrier pipeline fed by one producer
// warp; consumer warps (16 query rows each) run QK^T and PV on mma.sync with
// an online softmax in fp32 (exp2 domain).  Long contexts are split across
// CTAs; a merge kernel combines the splits with their log-sum-exp weights.
#include <math.h>

#include "common.cuh"
#include "launch.cuh"

namespace spec {

namespace {

constexpr int kAttnStages = 3;
constexpr int kMaxRowTiles = 4;  // up to 64 query rows (W * group) per CTA

template <int HD>
struct AttnCfg {
  static constexpr int kHalves = HD / 64;
  static constexpr int kTileBytes = kPage * HD * 2;  // one K (or V) page of one kv head
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kSmemBytes = kAttnStages * kStageBytes + 2 * kAttnStages * 8 + 1024;
};

template <int HD>
__global__ void __launch_bounds__((kMaxRowTiles + 1) * 32)
    attention_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ AttnParams p) {
  using C = AttnCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kAttnStages * C::kStageBytes);
  uint64_t* empty = full + kAttnStages;

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_row_tiles = blockDim.x / 32 - 1;
  const int grp = p.Hq / p.Hkv;
  const int rows = p.W * grp;

  pdl_wait();
  pdl_launch_dependents();

  const int sid = p.seq_ids[b];
  const bool sid_ok = sid >= 0 && sid < p.max_batch;  // a bad id was flagged by the prepare kernel
  const int L = p.seq_start[b];
  const int n_keys = L + p.W;
  const int n_pages = sid_ok ? min((n_keys + kPage - 1) / kPage, p.max_pages) : 0;
  const int pg0 = split * p.pages_per_split;
  const int pg1 = min(pg0 + p.pages_per_split, n_pages);
  const int npg = max(0, pg1 - pg0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAttnStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], n_row_tiles);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == n_row_tiles) {
    // --------------------------------------------------------------- producer
    if (lane == 0 && npg > 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int32_t* pt = p.page_table + (long long)sid * p.max_pages;
      for (int i = 0; i < npg; ++i) {
        const int s = i % kAttnStages;
        const uint32_t use = i / kAttnStages;
        if (i >= kAttnStages && !mbar_wait(&empty[s], (use - 1) & 1, p.status)) break;
        int page = pt[pg0 + i];
        if (page < 0) {  // no page: read page 0 instead (the round is already flagged)
          set_status(p.status, SPEC_ERR_CAPACITY);
          page = 0;
        }
        const int row = p.layer_row0 + (page * p.Hkv + kvh) * kPage;
        uint8_t* st = smem + s * C::kStageBytes;
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
#pragma unroll
        for (int h = 0; h < C::kHalves; ++h) {
          tma_load_2d(st + h * (kPage * 128), &tmK, h * 64, row, &full[s]);
          tma_load_2d(st + C::kTileBytes + h * (kPage * 128), &tmV, h * 64, row, &full[s]);
        }
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int g = lane >> 2, c = lane & 3;
  // query rows of this thread: r0 = warp*16 + g, r1 = r0 + 8; row r -> window row j = r / grp
  int jrow[2], head[2];
  bool valid[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = warp * 16 + g + 8 * h;
    valid[h] = r < rows;
    jrow[h] = valid[h] ? r / grp : 0;
    head[h] = kvh * grp + (valid[h] ? r % grp : 0);
  }
  // Q fragments (A operand, rows x head_dim), straight from global (L2-resident)
  uint32_t qa[HD / 16][4];
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __nv_bfloat16* qr =
          p.q + ((long long)(b * p.W + jrow[h]) * p.Hq + head[h]) * HD + ks * 16 + 2 * c;
      const uint32_t lo = valid[h] ? *reinterpret_cast<const uint32_t*>(qr) : 0u;
      const uint32_t hi = valid[h] ? *reinterpret_cast<const uint32_t*>(qr + 8) : 0u;
      qa[ks][h] = lo;       // a0a1 (row g) / a2a3 (row g+8)
      qa[ks][2 + h] = hi;   // a4a5 / a6a7
    }
  }
  const uint32_t anc0 = valid[0] ? p.anc[jrow[0]] : 0u;
  const uint32_t anc1 = valid[1] ? p.anc[jrow[1]] : 0u;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);

  float acc[HD / 8][4];
#pragma unroll
  for (int t = 0; t < HD / 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY};
  float lrow[2] = {0.f, 0.f};

  bool ok = true;
  for (int i = 0; i < npg; ++i) {
    const int s = i % kAttnStages;
    const uint32_t use = i / kAttnStages;
    if (!mbar_wait(&full[s], use & 1, p.status)) {
      ok = false;
      break;
    }
    const uint32_t kbase = smem_u32(smem + s * C::kStageBytes);
    const uint32_t vbase = kbase + C::kTileBytes;

    // S = Q K^T for the page's 64 keys: 8 key tiles of 8
    float sc[8][4];
#pragma unroll
    for (int t = 0; t < 8; ++t) sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
      for (int tp = 0; tp < 4; ++tp) {
        const int key = tp * 16 + (lane & 7) + ((lane >> 4) & 1) * 8;
        const int d = ks * 16 + ((lane >> 3) & 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + (d >> 6) * (kPage * 128) + swz128(key, d & 63), b0, b1, b2, b3);
        mma_bf16_16816(sc[2 * tp], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        mma_bf16_16816(sc[2 * tp + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
      }
    }
    // mask + online softmax (exp2 domain)
    const int key0 = (pg0 + i) * kPage;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = e >> 1;
        const int tkey = key0 + t * 8 + 2 * c + (e & 1);
        const uint32_t anc = h ? anc1 : anc0;
        bool vis = tkey < L || (tkey < n_keys && ((anc >> (tkey - L)) & 1u));
        vis = vis && valid[h];
        const float v = vis ? sc[t][e] * scale_log2 : -INFINITY;
        sc[t][e] = v;
        mx[h] = fmaxf(mx[h], v);
      }
    }
    float alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      const float mnew = fmaxf(mrow[h], mx[h]);
      alpha[h] = (mrow[h] == -INFINITY) ? 0.f : exp2f(mrow[h] - mnew);
      mrow[h] = mnew;
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = e >> 1;
        const float pv = (mrow[h] == -INFINITY) ? 0.f : exp2f(sc[t][e] - mrow[h]);
        sc[t][e] = pv;
        rs[h] += pv;
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      rs[h] += __shfl_xor_sync(0xffffffffu, rs[h], 1);
      rs[h] += __shfl_xor_sync(0xffffffffu, rs[h], 2);
      lrow[h] = lrow[h] * alpha[h] + rs[h];
    }
#pragma unroll
    for (int t = 0; t < HD / 8; ++t) {
      acc[t][0] *= alpha[0];
      acc[t][1] *= alpha[0];
      acc[t][2] *= alpha[1];
      acc[t][3] *= alpha[1];
    }
    // O += P V: P from the score registers (bf16), V via transposed ldmatrix
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t a0 = pack_bf16x2(sc[2 * kk][0], sc[2 * kk][1]);
      const uint32_t a1 = pack_bf16x2(sc[2 * kk][2], sc[2 * kk][3]);
      const uint32_t a2 = pack_bf16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      const uint32_t a3 = pack_bf16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < HD / 16; ++dp) {
        const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int d = dp * 16 + ((lane >> 4) & 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(vbase + (d >> 6) * (kPage * 128) + swz128(key, d & 63), b0, b1, b2, b3);
        mma_bf16_16816(acc[2 * dp], a0, a1, a2, a3, b0, b1);
        mma_bf16_16816(acc[2 * dp + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (!ok) return;

  // partial results: unnormalised O, running max (log2 units) and sum
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (!valid[h]) continue;
    const long long rh = (long long)(b * p.W + jrow[h]) * p.Hq + head[h];
    float* o = p.part_acc + (rh * p.n_splits + split) * HD;
#pragma unroll
    for (int t = 0; t < HD / 8; ++t) {
      o[t * 8 + 2 * c] = acc[t][2 * h];
      o[t * 8 + 2 * c + 1] = acc[t][2 * h + 1];
    }
    if (c == 0) {
      float* ml = p.part_ml + (rh * p.n_splits + split) * 2;
      ml[0] = mrow[h];
      ml[1] = lrow[h];
    }
  }
}

// out[row, head, :] = sum_s w_s acc_s / sum_s w_s l_s with w_s = 2^(m_s - max_s m_s)
template <int HD>
__global__ void __launch_bounds__(HD) attn_merge_kernel(const float* part_acc, const float* part_ml, int Hq,
                                                        int n_splits, __nv_bfloat16* out) {
  pdl_wait();
  pdl_launch_dependents();
  const long long rh = blockIdx.x;  // row * Hq + head
  const int d = threadIdx.x;
  const float* ml = part_ml + rh * n_splits * 2;
  float mmax = -INFINITY;
  for (int s = 0; s < n_splits; ++s) mmax = fmaxf(mmax, ml[2 * s]);
  float num = 0.f, den = 0.f;
  if (mmax != -INFINITY) {
    for (int s = 0; s < n_splits; ++s) {
      const float ms = ml[2 * s];
      if (ms == -INFINITY) continue;
      const float w = exp2f(ms - mmax);
      den += w * ml[2 * s + 1];
      num += w * part_acc[(rh * n_splits + s) * HD + d];
    }
  }
  out[rh * HD + d] = __float2bfloat16(den > 0.f ? num / den : 0.f);
}

template <int HD>
cudaError_t launch_attention_hd(const CUtensorMap* tmK, const CUtensorMap* tmV, const AttnParams& p,
                                cudaStream_t st) {
  using C = AttnCfg<HD>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(attention_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int rows = p.W * (p.Hq / p.Hkv);
  const int row_tiles = (rows + 15) / 16;
  if (row_tiles > kMaxRowTiles) return cudaErrorInvalidValue;
  dim3 grid(p.n_splits, p.Hkv, p.B);
  return launch_k(attention_kernel<HD>, grid, dim3((row_tiles + 1) * 32), C::kSmemBytes, st, *tmK, *tmV, p);
}

}  // namespace

cudaError_t launch_attention(const CUtensorMap* tmK, const CUtensorMap* tmV, const AttnParams& p, cudaStream_t st) {
  if (p.hd == 128) return launch_attention_hd<128>(tmK, tmV, p, st);
  if (p.hd == 64) return launch_attention_hd<64>(tmK, tmV, p, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_merge(const float* part_acc, const float* part_ml, int M, int Hq, int hd, int n_splits,
                              __nv_bfloat16* out, cudaStream_t st) {
  dim3 grid(M * Hq);
  if (hd == 128) return launch_k(attn_merge_kernel<128>, grid, dim3(128), 0, st, part_acc, part_ml, Hq, n_splits, out);
  if (hd == 64) return launch_k(attn_merge_kernel<64>, grid, dim3(64), 0, st, part_acc, part_ml, Hq, n_splits, out);
  return cudaErrorInvalidValue;
}

}  // namespace spec
