// Skinny weight-streaming projection Y = X W^T for the verify forward, with the
// projection's epilogue fused in.
//
// The verify round's cost is the weight stream: every weight matrix is read
// from HBM once for all B*(gamma+1) rows ("Per-step cost versus accepted
// tokens", "Why a guess is worth anything": the step moves every weight once,
// however many positions it scores; Lecture 6 "Optimizing Autoregressive
// Decode" section 9.1: ~129 tokens ride in the shadow of the weight read at
// batch 1).  So the kernel is built around the weight stream:
//   * one producer warp drives a multi-stage TMA pipeline of 128 x 64 bf16
//     weight tiles (128-byte swizzle, L2 evict-first) plus the matching BM x 64
//     activation tile, completing on mbarriers;
//   * eight consumer warps each own 16 weight rows and run mma.sync m16n8k16
//     with the weights as the A operand ("swap-AB": weight rows on the MMA M
//     side, token rows on N, so 1..64 tokens need no padding to 64);
//   * split-K over gridDim.y fills the 152 SMs when N/128 tiles are few.  Each
//     split writes its fp32 partial tile; the last split CTA of a tile to
//     arrive (atomic tile counter, reset by that CTA) sums the partials in
//     split order -- deterministic -- and applies the epilogue;
//   * the weight prefetch is issued before griddepcontrol.wait, so under
//     programmatic dependent launch it overlaps the previous kernel's tail.
//
// RMSNorm is folded in: the producer of a normalised input stores
// X' = bf16(r * g) and per-128-column partial sums of r^2; the consumer scales
// each output row by s_m = rsqrt(sum r^2 / d + eps), since
// sum_k (s_m r_mk g_k) W_nk = s_m sum_k (r_mk g_k) W_nk.
#include <algorithm>

#include "common.cuh"
#include "launch.cuh"

namespace spec {

namespace {

constexpr int kBN = 128;          // weight rows per CTA
constexpr int kBK = 64;           // k per stage: one 128-byte swizzle row
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kTilePad = kBN + 4;  // fp32 epilogue tile row pitch

template <int BM>
struct GemmCfg {
  static constexpr int kStages = BM <= 16 ? 6 : 4;
  static constexpr int kWBytes = kBN * kBK * 2;
  static constexpr int kXBytes = BM * kBK * 2;
  static constexpr int kStageBytes = kWBytes + kXBytes;
  static constexpr int kPipeBytes = kStages * kStageBytes;
  static constexpr int kTileBytes = BM * kTilePad * 4;
  static_assert(kTileBytes <= kPipeBytes, "epilogue tile reuses the pipeline buffers");
  static constexpr int kSmemBytes = kPipeBytes + 2 * kStages * 8 + BM * 4 + 1024;
};

SPEC_DEVICE_INLINE void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

template <int BM, int EPI>
__global__ void __launch_bounds__(kThreads, 2)
    gemm_swapab_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ EpiParams p) {
  using C = GemmCfg<BM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kPipeBytes);
  uint64_t* empty = full + C::kStages;
  float* s_scale = reinterpret_cast<float*>(empty + C::kStages);
  __shared__ int s_last, s_fail;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBN;
  const int split = blockIdx.y;
  const int m0 = blockIdx.z * BM;
  const int kb0 = split * p.kb_per_split;
  const int nkb = min(p.kb_per_split, p.kb_total - kb0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    s_fail = 0;
    fence_barrier_init();
  }
  __syncthreads();

  auto stage_w = [&](int s) { return smem + s * C::kStageBytes; };
  auto stage_x = [&](int s) { return smem + s * C::kStageBytes + C::kWBytes; };

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nkb > 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmX);
      const uint64_t pol = l2_policy_evict_first();
      const int pre = min(nkb, C::kStages);
      for (int kb = 0; kb < pre; ++kb) {  // weights never depend on the previous kernel
        mbar_arrive_expect_tx(&full[kb], C::kStageBytes);
        tma_load_2d_hint(stage_w(kb), &tmW, (kb0 + kb) * kBK, n0, &full[kb], pol);
      }
      pdl_wait();
      pdl_launch_dependents();
      for (int kb = 0; kb < pre; ++kb) tma_load_2d(stage_x(kb), &tmX, (kb0 + kb) * kBK, m0, &full[kb]);
      for (int kb = pre; kb < nkb; ++kb) {
        const int s = kb % C::kStages;
        const uint32_t use = kb / C::kStages;
        if (!mbar_wait(&empty[s], (use - 1) & 1, p.status)) break;
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
        tma_load_2d_hint(stage_w(s), &tmW, (kb0 + kb) * kBK, n0, &full[s], pol);
        tma_load_2d(stage_x(s), &tmX, (kb0 + kb) * kBK, m0, &full[s]);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x;  // 0..255
  float acc[BM / 8][4];
#pragma unroll
  for (int t = 0; t < BM / 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  const int wrow = warp * 16;
  bool ok = true;
  for (int kb = 0; kb < nkb; ++kb) {
    const int s = kb % C::kStages;
    const uint32_t use = kb / C::kStages;
    if (!mbar_wait(&full[s], use & 1, p.status)) {
      ok = false;
      break;
    }
    const uint32_t wbase = smem_u32(stage_w(s));
    const uint32_t xbase = smem_u32(stage_x(s));
#pragma unroll
    for (int kk = 0; kk < kBK / 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      const int arow = wrow + (lane & 7) + ((lane >> 3) & 1) * 8;
      const int acol = kk * 16 + (lane >> 4) * 8;
      ldsm_x4(wbase + swz128(arow, acol), a0, a1, a2, a3);
      if constexpr (BM == 8) {
        uint32_t b0, b1;
        const int brow = lane & 7;
        const int bcol = kk * 16 + ((lane >> 3) & 1) * 8;
        ldsm_x2(xbase + swz128(brow, bcol), b0, b1);
        mma_bf16_16816(acc[0], a0, a1, a2, a3, b0, b1);
      } else {
#pragma unroll
        for (int nt = 0; nt < BM / 16; ++nt) {
          uint32_t b0, b1, b2, b3;
          const int brow = nt * 16 + (lane & 7) + ((lane >> 4) & 1) * 8;
          const int bcol = kk * 16 + ((lane >> 3) & 1) * 8;
          ldsm_x4(xbase + swz128(brow, bcol), b0, b1, b2, b3);
          mma_bf16_16816(acc[2 * nt], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(acc[2 * nt + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  // A bounded wait that ran out in any consumer warp makes all of them return
  // (block-uniform decision) without touching outputs; the status word says why.
  const int g = lane >> 2, c = lane & 3;
  float* tile = reinterpret_cast<float*>(smem);  // reuses the (now idle) pipeline buffers
  if (!ok) s_fail = 1;
  consumer_sync();
  if (s_fail) return;

  // acc[t] = D tile (16 weight rows x 8 tokens): d0,d1 -> (row g, tokens 2c, 2c+1),
  // d2,d3 -> (row g+8, same tokens).  Rows of the output tile = tokens.
  if (p.splits == 1) {
#pragma unroll
    for (int t = 0; t < BM / 8; ++t) {
      const int ml = t * 8 + 2 * c;
      tile[ml * kTilePad + wrow + g] = acc[t][0];
      tile[ml * kTilePad + wrow + g + 8] = acc[t][2];
      tile[(ml + 1) * kTilePad + wrow + g] = acc[t][1];
      tile[(ml + 1) * kTilePad + wrow + g + 8] = acc[t][3];
    }
  } else {
    float* out = p.part + (long long)split * p.split_stride;
    const int n = n0 + wrow + g;
#pragma unroll
    for (int t = 0; t < BM / 8; ++t) {
      const int m = m0 + t * 8 + 2 * c;
      if (m < p.M) {
        out[(long long)m * p.N + n] = acc[t][0];
        out[(long long)m * p.N + n + 8] = acc[t][2];
      }
      if (m + 1 < p.M) {
        out[(long long)(m + 1) * p.N + n] = acc[t][1];
        out[(long long)(m + 1) * p.N + n + 8] = acc[t][3];
      }
    }
    __threadfence();
    consumer_sync();
    if (tid == 0) {
      const int tile_id = blockIdx.z * gridDim.x + blockIdx.x;
      const int prev = atomicAdd(&p.counters[tile_id], 1);
      s_last = prev == p.splits - 1;
      if (s_last) p.counters[tile_id] = 0;  // ready for the next launch
    }
    consumer_sync();
    if (!s_last) return;
    __threadfence();
    // sum the partials in split order (deterministic whichever CTA is last)
    for (int e = tid; e < BM * kBN; e += kConsumers) {
      const int ml = e / kBN, cl = e % kBN;
      const int m = m0 + ml;
      float v = 0.f;
      if (m < p.M) {
        const float* src = p.part + (long long)m * p.N + n0 + cl;
        for (int s = 0; s < p.splits; ++s) v += __ldcg(src + s * p.split_stride);
      }
      tile[ml * kTilePad + cl] = v;
    }
  }
  // per-row scale of a normalised input: s_m = rsqrt(sum_t ssq[t][m] / d + eps)
  if (tid < BM) {
    float sc = 1.f;
    const int m = m0 + tid;
    if (p.ssq_in && m < p.M) {
      float ss = 0.f;
      for (int t = 0; t < p.ssq_tiles; ++t) ss += __ldcg(p.ssq_in + (long long)t * p.ssq_stride + m);
      sc = rsqrtf(ss * p.inv_d + p.eps);
    }
    s_scale[tid] = sc;
  }
  consumer_sync();

  if constexpr (EPI == kEpiQKV) {
    // tile = 128 fused-QKV columns (one head of 128, or two of 64); RoPE pairs (i, i + hd/2)
    const int half = p.hd >> 1;
    for (int e = tid; e < BM * (kBN / 2); e += kConsumers) {
      const int ml = e / (kBN / 2), pr = e % (kBN / 2);
      const int m = m0 + ml;
      if (m >= p.M) continue;
      const int cl = (pr / half) * p.hd + pr % half;
      const int n = n0 + cl;
      const int head = n / p.hd, i = n % p.hd;
      const float sc = s_scale[ml];
      float a = tile[ml * kTilePad + cl] * sc;
      float b = tile[ml * kTilePad + cl + half] * sc;
      if (head < p.Hq + p.Hkv) {
        const int pos = p.row_pos[m];
        const float cs = p.rope_cos[(long long)pos * half + i];
        const float sn = p.rope_sin[(long long)pos * half + i];
        const float ra = a * cs - b * sn;
        const float rb = a * sn + b * cs;
        a = ra;
        b = rb;
      }
      if (head < p.Hq) {
        __nv_bfloat16* q = p.q_out + ((long long)m * p.Hq + head) * p.hd;
        q[i] = __float2bfloat16(a);
        q[i + half] = __float2bfloat16(b);
      } else {
        const int slot = p.row_slot[m];
        if (slot < 0) continue;  // the round failed to get a page for this row
        const bool is_k = head < p.Hq + p.Hkv;
        const int kvh = is_k ? head - p.Hq : head - p.Hq - p.Hkv;
        __nv_bfloat16* dst =
            (is_k ? p.kpool : p.vpool) + (((long long)(slot / kPage) * p.Hkv + kvh) * kPage + slot % kPage) * p.hd;
        dst[i] = __float2bfloat16(a);
        dst[i + half] = __float2bfloat16(b);
      }
    }
  } else if constexpr (EPI == kEpiSwiGLU) {
    // tile = 64 gate rows then the 64 up rows of the same features
    const int f0 = (n0 / kBN) * 64;
    for (int e = tid; e < BM * 64; e += kConsumers) {
      const int ml = e / 64, fl = e % 64;
      const int m = m0 + ml;
      if (m >= p.M) continue;
      const float sc = s_scale[ml];
      const float gv = tile[ml * kTilePad + fl] * sc;
      const float uv = tile[ml * kTilePad + 64 + fl] * sc;
      const float silu = gv / (1.f + expf(-gv));
      p.act[(long long)m * p.ffn + f0 + fl] = __float2bfloat16(silu * uv);
    }
  } else if constexpr (EPI == kEpiResid) {
    // r += y; next input X' = bf16(r * g_next); per-tile sum of r^2 for the next norm.
    // Warp w handles rows w, w+8, ...; lane covers columns lane + 32j (fixed order).
    for (int ml = warp; ml < BM; ml += kConsumerWarps) {
      const int m = m0 + ml;
      if (m >= p.M) continue;
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < kBN / 32; ++j) {
        const int cl = lane + 32 * j;
        const long long idx = (long long)m * p.d + n0 + cl;
        const float r = p.resid[idx] + tile[ml * kTilePad + cl] * s_scale[ml];
        p.resid[idx] = r;
        p.xn[idx] = __float2bfloat16(r * p.g_next[n0 + cl]);
        ss += r * r;
      }
      ss = warp_sum(ss);
      if (lane == 0) p.ssq_out[(long long)(n0 / kBN) * p.ssq_stride + m] = ss;
    }
  } else {  // kEpiLogits: logits = s_m * y, plus per-tile softmax statistics of each row
    for (int ml = warp; ml < BM; ml += kConsumerWarps) {
      const int m = m0 + ml;
      if (m >= p.M) continue;
      const float sc = s_scale[ml];
      float v[kBN / 32];
      float mx = -INFINITY;
      int am = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < kBN / 32; ++j) {
        const int cl = lane + 32 * j;
        v[j] = tile[ml * kTilePad + cl] * sc;
        p.logits[(long long)m * p.N + n0 + cl] = v[j];
        if (v[j] > mx || (v[j] == mx && n0 + cl < am)) {
          mx = v[j];
          am = n0 + cl;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, mx, o);
        const int oa = __shfl_xor_sync(0xffffffffu, am, o);
        if (om > mx || (om == mx && oa < am)) {
          mx = om;
          am = oa;
        }
      }
      float se = 0.f;
      if (p.tstat_sum) {
#pragma unroll
        for (int j = 0; j < kBN / 32; ++j) se += expf((v[j] - mx) * p.inv_temp);
        se = warp_sum(se);
      }
      if (lane == 0) {
        const long long si = (long long)(n0 / kBN) * p.tstat_stride + m;
        p.tstat_max[si] = mx;
        p.tstat_arg[si] = am;
        if (p.tstat_sum) p.tstat_sum[si] = se;
      }
    }
  }
}

template <int BM, int EPI>
cudaError_t launch_bm(const CUtensorMap* tmW, const CUtensorMap* tmX, const EpiParams& p, cudaStream_t st) {
  using C = GemmCfg<BM>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemm_swapab_kernel<BM, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(p.N / kBN, p.splits, (p.M + BM - 1) / BM);
  return launch_k(gemm_swapab_kernel<BM, EPI>, grid, dim3(kThreads), C::kSmemBytes, st, *tmW, *tmX, p);
}

template <int EPI>
cudaError_t launch_epi(const CUtensorMap* tmW, const CUtensorMap* tmX, int BM, const EpiParams& p,
                       cudaStream_t st) {
  switch (BM) {
    case 8: return launch_bm<8, EPI>(tmW, tmX, p, st);
    case 16: return launch_bm<16, EPI>(tmW, tmX, p, st);
    case 32: return launch_bm<32, EPI>(tmW, tmX, p, st);
    case 64: return launch_bm<64, EPI>(tmW, tmX, p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int choose_bm(int M) {
  if (M <= 8) return 8;
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  return 64;
}

int choose_splits(int N, int K, int M, int BM, int sm_count, int max_splits) {
  // One wave: at most two CTAs per SM (the shared-memory limit), so every split of
  // a tile is resident at once and no tile's reduction waits for a second wave.
  const int tiles = (N / kBN) * ((M + BM - 1) / BM);
  const int kb = K / kBK;
  const int slots = 2 * sm_count;
  int s = std::max(1, slots / tiles);
  s = std::min(s, std::min(max_splits, std::max(1, kb / 4)));
  const int per = (kb + s - 1) / s;  // make every split non-empty
  return (kb + per - 1) / per;
}

cudaError_t launch_gemm_epi(int epi, const CUtensorMap* tmW, const CUtensorMap* tmX, int BM, EpiParams p,
                            cudaStream_t st) {
  p.kb_total = p.K / kBK;
  p.kb_per_split = (p.kb_total + p.splits - 1) / p.splits;
  switch (epi) {
    case kEpiQKV: return launch_epi<kEpiQKV>(tmW, tmX, BM, p, st);
    case kEpiSwiGLU: return launch_epi<kEpiSwiGLU>(tmW, tmX, BM, p, st);
    case kEpiResid: return launch_epi<kEpiResid>(tmW, tmX, BM, p, st);
    case kEpiLogits: return launch_epi<kEpiLogits>(tmW, tmX, BM, p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace spec
