// Skinny weight-streaming projection Y = X W^T for the verify forward, with the
// projection's epilogue fused in.
//
// The verify round's cost is the weight stream: every weight matrix is read
// from HBM once for all B*(gamma+1) rows ("Per-step cost versus accepted
// tokens", "Why a guess is worth anything": the step moves every weight once,
// however many positions it scores; Lecture 6 "Optimizing Autoregressive
// Decode" section 9.1: ~129 tokens ride in the shadow of the weight read at
// batch 1).  So the kernel is built around the weight stream:
//   * one producer warp drives a multi-stage TMA pipeline of 128 x 64 fp16
//     weight tiles (the bf16 weights re-encoded exactly as fp16 x 2^e per row) (128-byte swizzle, L2 evict-first) plus the matching BM x 64
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
// X' = fp16(r * g) and per-128-column partial sums of r^2; the consumer scales
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

template <int N>
SPEC_DEVICE_INLINE void named_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

// The end of a tile, common to both projection kernels.  Called by the NT
// epilogue threads (tid 0..NT-1, warp = tid / 32) once this CTA's accumulator is
// in `tile` (splits == 1) or its partial is in p.part (splits > 1).  With split-K
// the last CTA of the tile to arrive reduces the partials in split order, the
// others return.  Then the row scales and the projection's epilogue.
template <int EPI, int NT, int ROWS>
SPEC_DEVICE_INLINE void finish_tile(const EpiParams& p, float* tile, float* s_scale, int* s_last, int m0, int n0,
                                    int tid, int warp, int lane) {
  constexpr int kGroupWarps = NT / 32;
  if (p.splits > 1) {
    __threadfence();
    named_sync<NT>();
    if (tid == 0) {
      const int tile_id = blockIdx.z * gridDim.x + blockIdx.x;
      const int prev = atomicAdd(&p.counters[tile_id], 1);
      *s_last = prev == p.splits - 1;
      if (*s_last) p.counters[tile_id] = 0;  // ready for the next launch
    }
    named_sync<NT>();
    if (!*s_last) return;
    __threadfence();
    // sum the partials in split order (deterministic whichever CTA is last);
    // 4 columns per thread, partials of 4 splits loaded before they are added
    for (int e = tid; e < ROWS * (kBN / 4); e += NT) {
      const int ml = e / (kBN / 4), cl = (e % (kBN / 4)) * 4;
      const int m = m0 + ml;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (m < p.M) {
        const float* src = p.part + (long long)m * p.N + n0 + cl;
        int s = 0;
        for (; s + 4 <= p.splits; s += 4) {
          float4 a[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) a[j] = __ldcg(reinterpret_cast<const float4*>(src + (s + j) * p.split_stride));
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            v.x += a[j].x;
            v.y += a[j].y;
            v.z += a[j].z;
            v.w += a[j].w;
          }
        }
        for (; s < p.splits; ++s) {
          const float4 a = __ldcg(reinterpret_cast<const float4*>(src + s * p.split_stride));
          v.x += a.x;
          v.y += a.y;
          v.z += a.z;
          v.w += a.w;
        }
      }
      *reinterpret_cast<float4*>(&tile[ml * kTilePad + cl]) = v;
    }
  }
  // weight-row scale 2^-e of the fp16 encoding, per output column of the tile
  __shared__ float s_rs[kBN];
  for (int cl = tid; cl < kBN; cl += NT) s_rs[cl] = p.rscale[n0 + cl];
  // per-row scale of a normalised input: s_m = rsqrt(sum_t ssq[t][m] / d + eps).
  // One warp per row, one tile partial per lane (independent loads, then a fixed
  // shuffle tree: the same order on every run).
#pragma unroll 4
  for (int r = warp; r < ROWS; r += kGroupWarps) {
    const int m = m0 + r;
    float sc = 1.f;
    if (p.ssq_in && m < p.M) {
      float ss = 0.f;
      for (int t = lane; t < p.ssq_tiles; t += 32) ss += __ldcg(p.ssq_in + (long long)t * p.ssq_stride + m);
      ss = warp_sum(ss);
      sc = rsqrtf(ss * p.inv_d + p.eps);
    }
    if (lane == 0) s_scale[r] = sc;
  }
  named_sync<NT>();

  if constexpr (EPI == kEpiQKV) {
    // tile = 128 fused-QKV columns (one head of 128, or two of 64); RoPE pairs (i, i + hd/2)
    const int half = p.hd >> 1;
    for (int e = tid; e < ROWS * (kBN / 2); e += NT) {
      const int ml = e / (kBN / 2), pr = e % (kBN / 2);
      const int m = m0 + ml;
      if (m >= p.M) continue;
      const int cl = (pr / half) * p.hd + pr % half;
      const int n = n0 + cl;
      const int head = n / p.hd, i = n % p.hd;
      const float sc = s_scale[ml];
      float a = tile[ml * kTilePad + cl] * (sc * s_rs[cl]);
      float b = tile[ml * kTilePad + cl + half] * (sc * s_rs[cl + half]);
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
        act_t* q = p.q_out + ((long long)m * p.Hq + head) * p.hd;
        q[i] = to_act(a);
        q[i + half] = to_act(b);
      } else {
        const int slot = p.row_slot[m];
        if (slot < 0) continue;  // the round failed to get a page for this row
        const bool is_k = head < p.Hq + p.Hkv;
        const int kvh = is_k ? head - p.Hq : head - p.Hq - p.Hkv;
        act_t* dst =
            (is_k ? p.kpool : p.vpool) + (((long long)(slot / kPage) * p.Hkv + kvh) * kPage + slot % kPage) * p.hd;
        dst[i] = to_act(a);
        dst[i + half] = to_act(b);
      }
    }
  } else if constexpr (EPI == kEpiSwiGLU) {
    // tile = 64 gate rows then the 64 up rows of the same features
    const int f0 = (n0 / kBN) * 64;
    for (int e = tid; e < ROWS * 64; e += NT) {
      const int ml = e / 64, fl = e % 64;
      const int m = m0 + ml;
      if (m >= p.M) continue;
      const float sc = s_scale[ml];
      const float gv = tile[ml * kTilePad + fl] * (sc * s_rs[fl]);
      const float uv = tile[ml * kTilePad + 64 + fl] * (sc * s_rs[64 + fl]);
      const float silu = gv / (1.f + expf(-gv));
      p.act[(long long)m * p.ffn + f0 + fl] = to_act(silu * uv);
    }
  } else if constexpr (EPI == kEpiResid) {
    // r += y; next input X' = fp16(r * g_next); per-tile sum of r^2 for the next norm.
    // Warp w handles rows w, w+8, ...; lane covers columns lane + 32j (fixed order).
    for (int ml = warp; ml < ROWS; ml += kGroupWarps) {
      const int m = m0 + ml;
      if (m >= p.M) continue;
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < kBN / 32; ++j) {
        const int cl = lane + 32 * j;
        const long long idx = (long long)m * p.d + n0 + cl;
        const float r = p.resid[idx] + tile[ml * kTilePad + cl] * (s_scale[ml] * s_rs[cl]);
        p.resid[idx] = r;
        p.xn[idx] = to_act(r * p.g_next[n0 + cl]);
        ss += r * r;
      }
      ss = warp_sum(ss);
      if (lane == 0) p.ssq_out[(long long)(n0 / kBN) * p.ssq_stride + m] = ss;
    }
  } else {  // kEpiLogits: logits = s_m * y, plus per-tile softmax statistics of each row
    for (int ml = warp; ml < ROWS; ml += kGroupWarps) {
      const int m = m0 + ml;
      if (m >= p.M) continue;
      const float sc = s_scale[ml];
      float v[kBN / 32];
      float mx = -INFINITY;
      int am = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < kBN / 32; ++j) {
        const int cl = lane + 32 * j;
        v[j] = tile[ml * kTilePad + cl] * (sc * s_rs[cl]);
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
        mma_f16_16816(acc[0], a0, a1, a2, a3, b0, b1);
      } else {
#pragma unroll
        for (int nt = 0; nt < BM / 16; ++nt) {
          uint32_t b0, b1, b2, b3;
          const int brow = nt * 16 + (lane & 7) + ((lane >> 4) & 1) * 8;
          const int bcol = kk * 16 + ((lane >> 3) & 1) * 8;
          ldsm_x4(xbase + swz128(brow, bcol), b0, b1, b2, b3);
          mma_f16_16816(acc[2 * nt], a0, a1, a2, a3, b0, b1);
          mma_f16_16816(acc[2 * nt + 1], a0, a1, a2, a3, b2, b3);
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
  named_sync<kConsumers>();
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
  }
  finish_tile<EPI, kConsumers, BM>(p, tile, s_scale, &s_last, m0, n0, tid, warp, lane);
}


// ----------------------------------------------------------------------------
// tcgen05 path for more than 16 token rows: the same weight stream, but the
// contraction runs on the 5th-generation tensor cores.  One CTA = 128 weight
// rows x NT token rows (NT in 32..256, so up to 256 rows stream each weight
// tile exactly once).  Warp 0 drives TMA, one thread of warp 1 issues
// tcgen05.mma (A = 128 weight rows, B = NT token rows, both K-major with the
// 128-byte swizzle, fp32 accumulator in TMEM) and commits each stage back to the
// producer; warps 2..5 read the accumulator out of TMEM (each warp its 32-lane
// quarter) and run the same tile finish as the mma.sync path.
constexpr int kTcThreads = 192;

template <int NT>
struct TcCfg {
  static constexpr int kStages = NT == 256 ? 4 : (NT == 128 ? 3 : (NT == 64 ? 4 : 5));
  static constexpr int kWBytes = kBN * kBK * 2;
  static constexpr int kXBytes = NT * kBK * 2;
  static constexpr int kStageBytes = kWBytes + kXBytes;
  static constexpr int kPipeBytes = kStages * kStageBytes;
  static constexpr int kTileBytes = NT * kTilePad * 4;
  static_assert(kTileBytes <= kPipeBytes, "epilogue tile reuses the pipeline buffers");
  static constexpr int kTmemCols = NT;  // fp32 accumulator: one column per token row
  static constexpr int kSmemBytes = kPipeBytes + (2 * kStages + 1) * 8 + 16 + NT * 4 + 1024;
};

template <int NT, int EPI>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ EpiParams p) {
  using C = TcCfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kPipeBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* accum = empty + C::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  float* s_scale = reinterpret_cast<float*>(tmem_slot + 4);
  __shared__ int s_last, s_fail;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBN;
  const int split = blockIdx.y;
  const int m0 = blockIdx.z * NT;
  const int kb0 = split * p.kb_per_split;
  const int nkb = min(p.kb_per_split, p.kb_total - kb0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    s_fail = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto stage_w = [&](int s) { return smem + s * C::kStageBytes; };
  auto stage_x = [&](int s) { return smem + s * C::kStageBytes + C::kWBytes; };

  if (warp == 0) {
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
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------- MMA issue (1 thread)
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kBN, NT);
      int kb = 0;
      for (; kb < nkb; ++kb) {
        const int s = kb % C::kStages;
        const uint32_t use = kb / C::kStages;
        if (!mbar_wait(&full[s], use & 1, p.status)) {
          s_fail = 1;
          break;
        }
        tc_fence_after();
        const uint32_t wb = smem_u32(stage_w(s)), xb = smem_u32(stage_x(s));
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          tc_mma(tmem, sdesc_k_sw128(wb + kk * 32), sdesc_k_sw128(xb + kk * 32), idesc, (kb | kk) != 0);
        tc_commit(&empty[s]);  // the stage is free once these MMAs have read it
      }
      if (nkb <= 0) s_fail = 1;
      tc_commit(accum);  // arrives when every MMA issued above has completed
    }
    __syncwarp();
  } else {
    // ----------------------------------- TMEM -> tile / partials (warps 2..5)
    pdl_wait();
    pdl_launch_dependents();
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int nl = q * 32 + lane;      // weight row of this thread within the tile
    const bool done = mbar_wait(accum, 0, p.status);
    tc_fence_after();
    if (!done) s_fail = 1;
    float* tile = reinterpret_cast<float*>(smem);  // MMAs and loads are done with the stages
    if (done) {
      float* out = p.part + (long long)split * p.split_stride;
#pragma unroll 1
      for (int c0 = 0; c0 < NT; c0 += 16) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
        if (p.splits == 1) {
#pragma unroll
          for (int i = 0; i < 16; ++i) tile[(c0 + i) * kTilePad + nl] = v[i];
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int m = m0 + c0 + i;
            if (m < p.M) out[(long long)m * p.N + n0 + nl] = v[i];
          }
        }
      }
    }
    tc_fence_before();
  }
  // All warps: the accumulator has been read out (or the round failed); free TMEM,
  // then every thread of the CTA finishes the tile.
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (s_fail) return;
  if (warp < 2) pdl_wait();  // outputs are written below by every warp
  finish_tile<EPI, kTcThreads, NT>(p, reinterpret_cast<float*>(smem), s_scale, &s_last, m0, n0, threadIdx.x, warp,
                                   lane);
}

template <int NT, int EPI>
cudaError_t launch_tc(const CUtensorMap* tmW, const CUtensorMap* tmX, const EpiParams& p, cudaStream_t st) {
  using C = TcCfg<NT>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_tc_kernel<NT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(p.N / kBN, p.splits, (p.M + NT - 1) / NT);
  return launch_k(gemm_tc_kernel<NT, EPI>, grid, dim3(kTcThreads), C::kSmemBytes, st, *tmW, *tmX, p);
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
  switch (BM) {  // up to 64 token rows: mma.sync (HBM-bound); above: tcgen05
    case 8: return launch_bm<8, EPI>(tmW, tmX, p, st);
    case 16: return launch_bm<16, EPI>(tmW, tmX, p, st);
    case 32: return launch_bm<32, EPI>(tmW, tmX, p, st);
    case 64: return launch_bm<64, EPI>(tmW, tmX, p, st);
    case 128: return launch_tc<128, EPI>(tmW, tmX, p, st);
    case 256: return launch_tc<256, EPI>(tmW, tmX, p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int choose_bm(int M) {
  if (M <= 8) return 8;
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
}

int choose_splits(int N, int K, int M, int BM, int sm_count, int max_splits) {
  // One wave: as many CTAs as fit at once (shared memory allows two per SM up to
  // 64 token rows, one above), so every split of a tile is resident together and
  // no tile's reduction waits for a second wave.
  const int tiles = (N / kBN) * ((M + BM - 1) / BM);
  const int kb = K / kBK;
  const int slots = (BM <= 128 ? 2 : 1) * sm_count;
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
