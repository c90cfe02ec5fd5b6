// Skinny weight-streaming projection Y = X W^T for the verify forward.
//
// The verify round's cost is the weight stream: every weight matrix is read
// from HBM once for all B*(gamma+1) rows ("Per-step cost versus accepted
// tokens", "Why a guess is worth anything": the step moves every weight once,
// however many positions it scores; Lecture 6 section 9.1: up to ~129 tokens
// ride in the shadow of the weight read at batch 1).  So the kernel is built
// around the weight stream:
//   * one producer warp drives a multi-stage TMA pipeline of 128 x 64 bf16
//     weight tiles (128-byte swizzle, L2 evict-first) plus the matching
//     BM x 64 activation tile, completing on mbarriers;
//   * eight consumer warps each own 16 weight rows and run mma.sync
//     m16n8k16 with the weights as the A operand ("swap-AB": weight rows on
//     the MMA M side, token rows on N, so 1..64 tokens need no padding to 64);
//   * split-K over gridDim.y fills the 152 SMs when N/128 tiles are few; the
//     partial sums land in an fp32 workspace that the next (elementwise)
//     kernel reduces in a fixed order, so results are deterministic.
//   * the weight prefetch is issued before griddepcontrol.wait, so under
//     programmatic dependent launch it overlaps the previous kernel's tail.
#include <algorithm>

#include "common.cuh"
#include "launch.cuh"

namespace spec {

namespace {

constexpr int kBN = 128;          // weight rows per CTA
constexpr int kBK = 64;           // k per stage: one 128-byte swizzle row
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

template <int BM>
struct GemmCfg {
  static constexpr int kStages = BM <= 16 ? 6 : 4;
  static constexpr int kWBytes = kBN * kBK * 2;
  static constexpr int kXBytes = BM * kBK * 2;
  static constexpr int kStageBytes = kWBytes + kXBytes;
  static constexpr int kSmemBytes = kStages * kStageBytes + 2 * kStages * 8 + 1024;
};

struct GemmParams {
  int M;
  int kb_total;
  int kb_per_split;
  float* out;
  long long split_stride;
  int ldo;
  int* status;
};

template <int BM>
__global__ void __launch_bounds__(kThreads, 2)
    gemm_swapab_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       GemmParams p) {
  using C = GemmCfg<BM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;

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
  if (!ok) return;

  // Epilogue: acc[t] = D tile (16 weight rows x 8 tokens); d0,d1 -> (row g, tokens 2c, 2c+1),
  // d2,d3 -> (row g+8, same tokens).
  float* out = p.out + (long long)split * p.split_stride;
  const int g = lane >> 2, c = lane & 3;
  const int n = n0 + wrow + g;
#pragma unroll
  for (int t = 0; t < BM / 8; ++t) {
    const int m = m0 + t * 8 + 2 * c;
    if (m < p.M) {
      out[(long long)m * p.ldo + n] = acc[t][0];
      out[(long long)m * p.ldo + n + 8] = acc[t][2];
    }
    if (m + 1 < p.M) {
      out[(long long)(m + 1) * p.ldo + n] = acc[t][1];
      out[(long long)(m + 1) * p.ldo + n + 8] = acc[t][3];
    }
  }
}

template <int BM>
cudaError_t launch_bm(const CUtensorMap* tmW, const CUtensorMap* tmX, int N, int K, int M, int splits, float* out,
                      long long split_stride, int ldo, int* status, cudaStream_t st) {
  using C = GemmCfg<BM>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemm_swapab_kernel<BM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  GemmParams p;
  p.M = M;
  p.kb_total = K / kBK;
  p.kb_per_split = (p.kb_total + splits - 1) / splits;
  p.out = out;
  p.split_stride = split_stride;
  p.ldo = ldo;
  p.status = status;
  dim3 grid(N / kBN, splits, (M + BM - 1) / BM);
  return launch_k(gemm_swapab_kernel<BM>, grid, dim3(kThreads), C::kSmemBytes, st, *tmW, *tmX, p);
}

}  // namespace

int choose_bm(int M) {
  if (M <= 8) return 8;
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  return 64;
}

int choose_splits(int N, int K, int M, int BM, int sm_count, int max_splits) {
  const int tiles = (N / kBN) * ((M + BM - 1) / BM);
  const int kb = K / kBK;
  const int target = 2 * sm_count;  // two CTAs resident per SM
  int s = (target + tiles - 1) / tiles;
  s = std::max(1, std::min(s, std::min(max_splits, kb / 4 > 0 ? kb / 4 : 1)));
  // make every split non-empty
  const int per = (kb + s - 1) / s;
  return (kb + per - 1) / per;
}

cudaError_t launch_gemm(const CUtensorMap* tmW, const CUtensorMap* tmX, int BM, int N, int K, int M, int splits,
                        float* out, long long split_stride, int ldo, int* status, cudaStream_t st) {
  switch (BM) {
    case 8: return launch_bm<8>(tmW, tmX, N, K, M, splits, out, split_stride, ldo, status, st);
    case 16: return launch_bm<16>(tmW, tmX, N, K, M, splits, out, split_stride, ldo, status, st);
    case 32: return launch_bm<32>(tmW, tmX, N, K, M, splits, out, split_stride, ldo, status, st);
    case 64: return launch_bm<64>(tmW, tmX, N, K, M, splits, out, split_stride, ldo, status, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace spec
