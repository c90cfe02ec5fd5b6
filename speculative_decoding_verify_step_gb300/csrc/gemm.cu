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
//     weight tiles (the bf16 weights re-encoded exactly as fp16 x 2^e per row;
//     128-byte swizzle, L2 evict-first) plus the matching BM x 64 activation
//     tile, completing on mbarriers, then prefetches the start of the next
//     projection's weights into L2;
//   * eight consumer warps each own 16 weight rows and run mma.sync m16n8k16
//     with the weights as the A operand ("swap-AB": weight rows on the MMA M
//     side, token rows on N, so 1..16 tokens need no padding to 64);
//   * split-K over gridDim.y fills the 152 SMs when N/128 tiles are few.  The
//     splits of a tile run as one thread-block cluster: each keeps its fp32
//     partial tile in its own shared memory, and after a cluster barrier split r
//     sums its share of the tile's rows over all splits through distributed
//     shared memory, in split order -- deterministic -- and applies the
//     epilogue to those rows;
//   * the weight prefetch is issued before griddepcontrol.wait, so under
//     programmatic dependent launch it overlaps the previous kernel's tail.
// This mma.sync kernel serves up to 16 token rows; from 17 rows the tcgen05
// kernel below takes over (tiles of 64 or 128 token rows).
//
// RMSNorm is folded in: the producer of a normalised input stores
// X' = fp16(r * g) and per-128-column partial sums of r^2; the consumer scales
// each output row by s_m = rsqrt(sum r^2 / d + eps), since
// sum_k (s_m r_mk g_k) W_nk = s_m sum_k (r_mk g_k) W_nk.
#include <algorithm>
#include <mutex>

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
constexpr int kMaxSplits = 16;     // split-K cluster size limit (non-portable above 8)

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

// Rows [r_lo, r_hi) of the token tile (at most `cap` rows from m0) that this CTA
// finishes: all of them, or with split-K the share of split blockIdx.y of the
// tile's real rows (a ragged tile of 80
// rows over 8 splits: 10 rows each, not 16 rows for five of them).
template <int ROWS>
SPEC_DEVICE_INLINE void tile_rows(const EpiParams& p, int m0, int& r_lo, int& r_hi, int cap = ROWS) {
  const int rows = max(0, min(cap, p.M - m0));
  r_lo = 0;
  r_hi = rows;
  if (p.splits > 1) {
    const int per = (rows + p.splits - 1) / p.splits;
    r_lo = min(rows, (int)blockIdx.y * per);
    r_hi = min(rows, r_lo + per);
  }
}

// Epilogue inputs that do not depend on the mainloop (weight-row scales, the
// input rows' sums of squares, the residual rows, RoPE angles, KV slots), loaded
// into registers before it so that their latency hides behind the weight stream.
// Token tiles of up to 16 rows only (measured: for 32 rows the extra registers
// spill, and wider tiles load them in the epilogue).
template <int EPI, int NT, int ROWS>
struct EpiPre {
  static constexpr bool kOn = ROWS <= 16;
  static constexpr int kWarps = NT / 32;
  static constexpr int kRowsW = (ROWS + kWarps - 1) / kWarps;       // rows per warp (warp-per-row loops)
  static constexpr int kPairs = (ROWS * (kBN / 2) + NT - 1) / NT;  // RoPE pairs per thread
  float rs;                 // weight-row scale of column tid (tid < kBN)
  float ssq[kRowsW][2];     // sum-of-squares tiles lane, lane + 32 of the warp's rows
  float res[kRowsW][4];     // kEpiResid: residual at (row, column lane + 32 j)
  float gn[4];              // kEpiResid: next gain of column lane + 32 j
  int slot[kPairs];         // kEpiQKV: KV slot, cos, sin of each pair of this thread
  float cs[kPairs], sn[kPairs];
};

template <int EPI, int NT, int ROWS>
SPEC_DEVICE_INLINE void epi_prefetch(const EpiParams& p, EpiPre<EPI, NT, ROWS>& pre, int m0, int n0, int tid,
                                     int warp, int lane) {
  using E = EpiPre<EPI, NT, ROWS>;
  if constexpr (E::kOn) {
    int r_lo, r_hi;
    tile_rows<ROWS>(p, m0, r_lo, r_hi);
    pre.rs = tid < kBN ? __ldg(p.rscale + n0 + tid) : 0.f;
#pragma unroll
    for (int k = 0; k < E::kRowsW; ++k) {
      const int r = r_lo + warp + k * E::kWarps;
      pre.ssq[k][0] = pre.ssq[k][1] = 0.f;
      if (r < r_hi && p.ssq_in) {
        const int m = m0 + r;
        if (lane < p.ssq_tiles) pre.ssq[k][0] = __ldcg(p.ssq_in + (long long)lane * p.ssq_stride + m);
        if (lane + 32 < p.ssq_tiles) pre.ssq[k][1] = __ldcg(p.ssq_in + (long long)(lane + 32) * p.ssq_stride + m);
      }
      if constexpr (EPI == kEpiResid) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          pre.res[k][j] = r < r_hi ? __ldcg(p.resid + (long long)(m0 + r) * p.d + n0 + lane + 32 * j) : 0.f;
      }
    }
    if constexpr (EPI == kEpiResid) {
#pragma unroll
      for (int j = 0; j < 4; ++j) pre.gn[j] = __ldg(p.g_next + n0 + lane + 32 * j);
    }
    if constexpr (EPI == kEpiQKV) {
      const int half = p.hd >> 1;
#pragma unroll
      for (int k = 0; k < E::kPairs; ++k) {
        const int e = tid + k * NT;
        pre.slot[k] = -1;
        pre.cs[k] = 1.f;
        pre.sn[k] = 0.f;
        if (e < max(0, r_hi - r_lo) * (kBN / 2)) {
          const int m = m0 + r_lo + e / (kBN / 2), pr = e % (kBN / 2);
          const int i = (n0 + (pr / half) * p.hd + pr % half) % p.hd;
          const int pos = __ldcg(p.row_pos + m);
          pre.slot[k] = __ldcg(p.row_slot + m);
          pre.cs[k] = __ldg(p.rope_cos + (long long)pos * half + i);
          pre.sn[k] = __ldg(p.rope_sin + (long long)pos * half + i);
        }
      }
    }
  }
}

// Split-K reduction of this split's rows: item e = (row r_lo + e / 32, columns
// 4 (e % 32) ..+3); each item sums the S CTAs' partials in split order (the same
// order on every run).  U items per thread are in flight at a time, their S
// remote loads each issued before any is used.
template <int S, int U, int NT>
SPEC_DEVICE_INLINE void reduce_rows(float* tile, int r_lo, int n_items, int tid, int rank0, int rstep) {
  for (int e0 = tid; e0 < n_items; e0 += U * NT) {
    float4 a[U][S];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = min(e0 + u * NT, n_items - 1);
      const uint32_t off = smem_u32(tile + (r_lo + e / (kBN / 4)) * kTilePad + (e % (kBN / 4)) * 4);
#pragma unroll
      for (int j = 0; j < S; ++j) a[u][j] = ld_dsmem_f4(mapa_u32(off, rank0 + j * rstep));
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = e0 + u * NT;
      if (e >= n_items) break;
      float4 v = a[u][0];
#pragma unroll
      for (int j = 1; j < S; ++j) {
        v.x += a[u][j].x;
        v.y += a[u][j].y;
        v.z += a[u][j].z;
        v.w += a[u][j].w;
      }
      *reinterpret_cast<float4*>(&tile[(r_lo + e / (kBN / 4)) * kTilePad + (e % (kBN / 4)) * 4]) = v;
    }
  }
}

template <int NT, int LOADS, int S = 2>
SPEC_DEVICE_INLINE void reduce_splits(int splits, float* tile, int r_lo, int n_items, int tid, int rank0 = 0,
                                      int rstep = 1) {
  if constexpr (LOADS == 1) {
    // one item at a time: a single loop for every split count (measured: the
    // specialised copies cost more in instruction fetch than they save here)
    for (int e = tid; e < n_items; e += NT) {
      const int ml = r_lo + e / (kBN / 4), cl = (e % (kBN / 4)) * 4;
      const uint32_t off = smem_u32(tile + ml * kTilePad + cl);
      float4 a[kMaxSplits];
#pragma unroll
      for (int j = 0; j < kMaxSplits; ++j)
        if (j < splits) a[j] = ld_dsmem_f4(mapa_u32(off, rank0 + j * rstep));
      float4 v = a[0];
#pragma unroll
      for (int j = 1; j < kMaxSplits; ++j)
        if (j < splits) {
          v.x += a[j].x;
          v.y += a[j].y;
          v.z += a[j].z;
          v.w += a[j].w;
        }
      *reinterpret_cast<float4*>(&tile[ml * kTilePad + cl]) = v;
    }
  } else if constexpr (S <= kMaxSplits) {
    if (splits == S) {
      reduce_rows<S, (LOADS / S > 1 ? LOADS / S : 1), NT>(tile, r_lo, n_items, tid, rank0, rstep);
    } else {
      reduce_splits<NT, LOADS, S + 1>(splits, tile, r_lo, n_items, tid, rank0, rstep);
    }
  }
}

// The end of a tile, common to both projection kernels.  Called by the NT
// epilogue threads (tid 0..NT-1, warp = tid / 32) once this CTA's accumulator is
// in `tile` (its own shared memory).  With split-K the splits of a tile form one
// thread-block cluster: after a cluster barrier, split r sums rows
// [r * ROWS/S, (r+1) * ROWS/S) of all S partial tiles through distributed shared
// memory, in split order (deterministic), and runs the epilogue on those rows --
// the reduction is spread over the S CTAs and never leaves the chip.  Split j's
// partial tile sits in the CTA of cluster rank rank0 + j * rstep (the CTA pairs of
// the pair kernel interleave their splits).  The caller holds back the CTA's exit
// with the matching cluster_wait().
//
// PREP: the weight-row scales, the row scales and (QKV) the rows' positions and
// KV slots were already placed in s_rs / s_scale / s_ps while the mainloop ran;
// LOADS: remote float4 loads of the split-K reduction in flight per thread.
template <int EPI, int NT, int ROWS, bool PREP = false, int LOADS = 1>
SPEC_DEVICE_INLINE void finish_tile(const EpiParams& p, const EpiPre<EPI, NT, ROWS>& pre, float* tile,
                                    float* s_scale, int m0, int n0, int tid, int warp, int lane,
                                    float* s_rs_prep = nullptr, const int2* s_ps = nullptr, int rank0 = 0,
                                    int rstep = 1, int rows_cap = ROWS) {
  using E = EpiPre<EPI, NT, ROWS>;
  constexpr int kGroupWarps = NT / 32;
  int r_lo, r_hi;
  tile_rows<ROWS>(p, m0, r_lo, r_hi, rows_cap);
  if (p.splits > 1) {
    cluster_arrive();  // this CTA's partial tile is written
    cluster_wait();    // ... and every other split's
    reduce_splits<NT, LOADS>(p.splits, tile, r_lo, max(0, r_hi - r_lo) * (kBN / 4), tid, rank0, rstep);
    __syncwarp();      // converged for the aligned cluster barrier
    cluster_arrive();  // done reading the other CTAs' tiles
  }
  // weight-row scale 2^-e of the fp16 encoding, per output column of the tile
  __shared__ __align__(16) float s_rs_own[kBN];
  float* s_rs = PREP ? s_rs_prep : s_rs_own;
  // per-row scale of a normalised input: s_m = rsqrt(sum_t ssq[t][m] / d + eps).
  // One warp per row, tiles lane, lane + 32, ... per lane (then a fixed shuffle
  // tree: the same order on every run).
  if constexpr (PREP) {
  } else if constexpr (E::kOn) {
    if (tid < kBN) s_rs[tid] = pre.rs;
#pragma unroll
    for (int k = 0; k < E::kRowsW; ++k) {
      const int r = r_lo + warp + k * kGroupWarps;
      if (r >= r_hi) break;
      float sc = 1.f;
      if (p.ssq_in) {
        float ss = pre.ssq[k][0] + pre.ssq[k][1];
        for (int t = lane + 64; t < p.ssq_tiles; t += 32) ss += __ldcg(p.ssq_in + (long long)t * p.ssq_stride + m0 + r);
        ss = warp_sum(ss);
        sc = rsqrtf(ss * p.inv_d + p.eps);
      }
      if (lane == 0) s_scale[r] = sc;
    }
  } else {
    for (int cl = tid; cl < kBN; cl += NT) s_rs[cl] = p.rscale[n0 + cl];
    // eight rows per warp at a time: their loads are issued together
    for (int r0 = r_lo + warp; r0 < r_hi; r0 += 8 * kGroupWarps) {
      float ss[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = r0 + j * kGroupWarps;
        float a = 0.f;
        if (r < r_hi && p.ssq_in)
          for (int t = lane; t < p.ssq_tiles; t += 32) a += __ldcg(p.ssq_in + (long long)t * p.ssq_stride + m0 + r);
        ss[j] = a;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = r0 + j * kGroupWarps;
        const float sum = warp_sum(ss[j]);
        if (r < r_hi && lane == 0) s_scale[r] = p.ssq_in ? rsqrtf(sum * p.inv_d + p.eps) : 1.f;
      }
    }
  }
  named_sync<NT>();

  if constexpr (EPI == kEpiQKV) {
    // tile = 128 fused-QKV columns (one head of 128, or two of 64); RoPE pairs (i, i + hd/2)
    const int half = p.hd >> 1;
    const int n_pairs = max(0, r_hi - r_lo) * (kBN / 2);
    auto pair = [&](int e, float cs, float sn, int slot) {
      const int ml = r_lo + e / (kBN / 2), pr = e % (kBN / 2);
      const int m = m0 + ml;
      const int cl = (pr / half) * p.hd + pr % half;
      const int n = n0 + cl;
      const int head = n / p.hd, i = n % p.hd;
      const float sc = s_scale[ml];
      float a = tile[ml * kTilePad + cl] * (sc * s_rs[cl]);
      float b = tile[ml * kTilePad + cl + half] * (sc * s_rs[cl + half]);
      if (head < p.Hq + p.Hkv) {
        const float ra = a * cs - b * sn;
        const float rb = a * sn + b * cs;
        a = ra;
        b = rb;
      }
      if (head < p.Hq) {
        act_t* q = p.q_out + ((long long)m * p.Hq + head) * p.hd;
        q[i] = to_act(a);
        q[i + half] = to_act(b);
      } else if (slot >= 0) {  // slot < 0: the round failed to get a page for this row
        const bool is_k = head < p.Hq + p.Hkv;
        const int kvh = is_k ? head - p.Hq : head - p.Hq - p.Hkv;
        act_t* dst =
            (is_k ? p.kpool : p.vpool) + (((long long)(slot / kPage) * p.Hkv + kvh) * kPage + slot % kPage) * p.hd;
        dst[i] = to_act(a);
        dst[i + half] = to_act(b);
      }
    };
    if constexpr (PREP) {
      // four consecutive pairs (i .. i+3 of one head) per item, two items per
      // thread at a time: their angles are loaded together, then written as
      // 8-byte groups (measured, 80-row tiles: batches of two finish the tile in
      // half the time of batches of eight, with the same loads)
      // head_dim is 64 or 128 and the tile starts on a head boundary (n0 is a
      // multiple of 128): pair pr of a row is element i = pr mod hd/2 of head
      // n0/hd + pr div hd/2, the divisions done as shifts and masks
      const int lh = 31 - __clz(p.hd);
      const int hmask = half - 1;
      const int head0 = n0 >> lh;
      const int n_quads = n_pairs / 4;
      constexpr int kB = 2;
      for (int e0 = tid; e0 < n_quads; e0 += kB * NT) {
        float4 cs[kB], sn[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const unsigned e = (unsigned)min(e0 + j * NT, n_quads - 1);
          const int ml = r_lo + (int)(e / (kBN / 8)), pr = (int)(e % (kBN / 8)) * 4;
          const long long a = (long long)s_ps[ml].x * half + (pr & hmask);
          cs[j] = __ldg(reinterpret_cast<const float4*>(p.rope_cos + a));
          sn[j] = __ldg(reinterpret_cast<const float4*>(p.rope_sin + a));
        }
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const unsigned e = (unsigned)(e0 + j * NT);
          if (e >= (unsigned)n_quads) break;
          const int ml = r_lo + (int)(e / (kBN / 8)), pr = (int)(e % (kBN / 8)) * 4;
          const int m = m0 + ml;
          const int hl = pr >> (lh - 1), i = pr & hmask;
          const int cl = (hl << lh) + i;
          const int head = head0 + hl;
          const float sc = s_scale[ml];
          const float4 ta = *reinterpret_cast<const float4*>(&tile[ml * kTilePad + cl]);
          const float4 tb = *reinterpret_cast<const float4*>(&tile[ml * kTilePad + cl + half]);
          const float4 ra = *reinterpret_cast<const float4*>(&s_rs[cl]);
          const float4 rb = *reinterpret_cast<const float4*>(&s_rs[cl + half]);
          float av[4] = {ta.x * (sc * ra.x), ta.y * (sc * ra.y), ta.z * (sc * ra.z), ta.w * (sc * ra.w)};
          float bv[4] = {tb.x * (sc * rb.x), tb.y * (sc * rb.y), tb.z * (sc * rb.z), tb.w * (sc * rb.w)};
          if (head < p.Hq + p.Hkv) {
            const float c4[4] = {cs[j].x, cs[j].y, cs[j].z, cs[j].w};
            const float s4[4] = {sn[j].x, sn[j].y, sn[j].z, sn[j].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float x = av[k] * c4[k] - bv[k] * s4[k];
              const float y = av[k] * s4[k] + bv[k] * c4[k];
              av[k] = x;
              bv[k] = y;
            }
          }
          act_t* dst = nullptr;
          if (head < p.Hq) {
            dst = p.q_out + ((long long)m * p.Hq + head) * p.hd;
          } else if (s_ps[ml].y >= 0) {  // slot < 0: the round failed to get a page for this row
            const unsigned slot = (unsigned)s_ps[ml].y;
            const bool is_k = head < p.Hq + p.Hkv;
            const int kvh = is_k ? head - p.Hq : head - p.Hq - p.Hkv;
            dst = (is_k ? p.kpool : p.vpool) +
                  ((((long long)(slot / kPage) * p.Hkv + kvh) * kPage + slot % kPage) << lh);
          }
          if (dst) {
            *reinterpret_cast<uint2*>(dst + i) = pack_act4(av[0], av[1], av[2], av[3]);
            *reinterpret_cast<uint2*>(dst + i + half) = pack_act4(bv[0], bv[1], bv[2], bv[3]);
          }
        }
      }
    } else if constexpr (E::kOn) {
#pragma unroll
      for (int k = 0; k < E::kPairs; ++k) {
        const int e = tid + k * NT;
        if (e < n_pairs) pair(e, pre.cs[k], pre.sn[k], pre.slot[k]);
      }
    } else {
      // four pairs per thread at a time: positions and slots, then the angles, are
      // loaded together before any of the four is written
      constexpr int kB = 4;
      for (int e0 = tid; e0 < n_pairs; e0 += kB * NT) {
        int pos[kB], slot[kB];
        float cs[kB], sn[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const int e = e0 + j * NT;
          const int m = m0 + r_lo + min(e, n_pairs - 1) / (kBN / 2);
          pos[j] = p.row_pos[m];
          slot[j] = p.row_slot[m];
        }
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const int pr = (e0 + j * NT) % (kBN / 2);
          const int i = (n0 + (pr / half) * p.hd + pr % half) % p.hd;
          cs[j] = p.rope_cos[(long long)pos[j] * half + i];
          sn[j] = p.rope_sin[(long long)pos[j] * half + i];
        }
#pragma unroll
        for (int j = 0; j < kB; ++j)
          if (e0 + j * NT < n_pairs) pair(e0 + j * NT, cs[j], sn[j], slot[j]);
      }
    }
  } else if constexpr (EPI == kEpiSwiGLU) {
    // tile = 64 gate rows then the 64 up rows of the same features; four
    // consecutive features of one row per item (16-byte tile reads, 8-byte stores)
    const int f0 = (n0 / kBN) * 64;
    const unsigned n_items = max(0, r_hi - r_lo) * 16;
    for (unsigned e = tid; e < n_items; e += NT) {
      const int ml = r_lo + (int)(e / 16), fl = (int)(e % 16) * 4;
      const int m = m0 + ml;
      const float sc = s_scale[ml];
      const float4 tg = *reinterpret_cast<const float4*>(&tile[ml * kTilePad + fl]);
      const float4 tu = *reinterpret_cast<const float4*>(&tile[ml * kTilePad + 64 + fl]);
      const float4 rg = *reinterpret_cast<const float4*>(&s_rs[fl]);
      const float4 ru = *reinterpret_cast<const float4*>(&s_rs[64 + fl]);
      const float g4[4] = {tg.x * (sc * rg.x), tg.y * (sc * rg.y), tg.z * (sc * rg.z), tg.w * (sc * rg.w)};
      const float u4[4] = {tu.x * (sc * ru.x), tu.y * (sc * ru.y), tu.z * (sc * ru.z), tu.w * (sc * ru.w)};
      float h[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) h[k] = g4[k] / (1.f + expf(-g4[k])) * u4[k];
      *reinterpret_cast<uint2*>(p.act + (long long)m * p.ffn + f0 + fl) = pack_act4(h[0], h[1], h[2], h[3]);
    }
  } else if constexpr (EPI == kEpiResid) {
    // r += y; next input X' = fp16(r * g_next); per-tile sum of r^2 for the next norm.
    // Warp w handles rows w, w+8, ...; lane covers columns lane + 32j (fixed order).
    auto row = [&](int ml, const float (&rin)[kBN / 32], const float (&gn)[kBN / 32]) {
      const int m = m0 + ml;
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < kBN / 32; ++j) {
        const int cl = lane + 32 * j;
        const long long idx = (long long)m * p.d + n0 + cl;
        const float r = rin[j] + tile[ml * kTilePad + cl] * (s_scale[ml] * s_rs[cl]);
        p.resid[idx] = r;
        p.xn[idx] = to_act(r * gn[j]);
        ss += r * r;
      }
      ss = warp_sum(ss);
      if (lane == 0) p.ssq_out[(long long)(n0 / kBN) * p.ssq_stride + m] = ss;
    };
    if constexpr (E::kOn) {
#pragma unroll
      for (int k = 0; k < E::kRowsW; ++k) {
        const int ml = r_lo + warp + k * kGroupWarps;
        if (ml >= r_hi) break;
        row(ml, pre.res[k], pre.gn);
      }
    } else {
      float gn[kBN / 32];
#pragma unroll
      for (int j = 0; j < kBN / 32; ++j) gn[j] = p.g_next[n0 + lane + 32 * j];
      // four (eight when the scales were prepared: registers are free) rows per
      // warp at a time: their residuals are loaded before any is written
      constexpr int kB = PREP ? 8 : 4;
      for (int r0 = r_lo + warp; r0 < r_hi; r0 += kB * kGroupWarps) {
        float rin[kB][kBN / 32];
#pragma unroll
        for (int k = 0; k < kB; ++k) {
          const int ml = min(r0 + k * kGroupWarps, r_hi - 1);
#pragma unroll
          for (int j = 0; j < kBN / 32; ++j) rin[k][j] = p.resid[(long long)(m0 + ml) * p.d + n0 + lane + 32 * j];
        }
#pragma unroll
        for (int k = 0; k < kB; ++k)
          if (r0 + k * kGroupWarps < r_hi) row(r0 + k * kGroupWarps, rin[k], gn);
      }
    }
  } else {  // kEpiLogits: logits = s_m * y, plus per-tile softmax statistics of each row
    for (int ml = r_lo + warp; ml < r_hi; ml += kGroupWarps) {
      const int m = m0 + ml;
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
  __shared__ int s_fail;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.z * kBN;
  const int split = blockIdx.y;
  const int m0 = blockIdx.x * BM;
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
      if (!p.late_dependents) pdl_launch_dependents();
      for (int kb = 0; kb < pre; ++kb) tma_load_2d(stage_x(kb), &tmX, (kb0 + kb) * kBK, m0, &full[kb]);
      for (int kb = pre; kb < nkb; ++kb) {
        const int s = kb % C::kStages;
        const uint32_t use = kb / C::kStages;
        if (!mbar_wait(&empty[s], (use - 1) & 1, p.status)) break;
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
        tma_load_2d_hint(stage_w(s), &tmW, (kb0 + kb) * kBK, n0, &full[s], pol);
        tma_load_2d(stage_x(s), &tmX, (kb0 + kb) * kBK, m0, &full[s]);
      }
      l2_prefetch_share(p.l2_next, p.l2_next_bytes);
    }
    __syncwarp();
    if (p.splits > 1) {  // the two cluster barriers of the split-K reduction
      cluster_arrive();
      cluster_wait();
      cluster_arrive();
      cluster_wait();
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();
  if (!p.late_dependents) pdl_launch_dependents();
  const int tid = threadIdx.x;  // 0..255
  EpiPre<EPI, kConsumers, BM> pre;
  epi_prefetch<EPI, kConsumers, BM>(p, pre, m0, n0, tid, warp, lane);
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
    // The stage is refilled by TMA (async proxy) after this arrive: order this
    // thread's ldmatrix reads (generic proxy) of it before that write.
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  // A bounded wait that ran out in any consumer warp makes all of them return
  // (block-uniform decision) without touching outputs; the status word says why.
  const int g = lane >> 2, c = lane & 3;
  float* tile = reinterpret_cast<float*>(smem);  // reuses the (now idle) pipeline buffers
  if (!ok) s_fail = 1;
  named_sync<kConsumers>();
  if (s_fail) {
    if (p.splits > 1) {  // still take part in the cluster barriers
      cluster_arrive();
      cluster_wait();
      cluster_arrive();
      cluster_wait();
    }
    return;
  }

  // acc[t] = D tile (16 weight rows x 8 tokens): d0,d1 -> (row g, tokens 2c, 2c+1),
  // d2,d3 -> (row g+8, same tokens).  Rows of the output tile = tokens.
#pragma unroll
  for (int t = 0; t < BM / 8; ++t) {
    const int ml = t * 8 + 2 * c;
    tile[ml * kTilePad + wrow + g] = acc[t][0];
    tile[ml * kTilePad + wrow + g + 8] = acc[t][2];
    tile[(ml + 1) * kTilePad + wrow + g] = acc[t][1];
    tile[(ml + 1) * kTilePad + wrow + g + 8] = acc[t][3];
  }
  named_sync<kConsumers>();
  finish_tile<EPI, kConsumers, BM>(p, pre, tile, s_scale, m0, n0, tid, warp, lane);
  if (p.late_dependents) pdl_launch_dependents();
  __syncwarp();
  if (p.splits > 1) cluster_wait();  // the other splits are done reading this CTA's tile
}


// ----------------------------------------------------------------------------
// tcgen05 path from 17 token rows: the same weight stream, but the contraction
// runs on the 5th-generation tensor cores.  One CTA = 128 weight rows x NT token
// rows (NT = 64 or 128; more rows take several token tiles, dispatched side by
// side so that one weight slab serves them from L2).  Warp 0 drives TMA, one
// thread of warp 1 issues tcgen05.mma (A = 128 weight rows, B = the tile's token
// rows, both K-major with the 128-byte swizzle, fp32 accumulator in TMEM) and
// commits each stage back to the producer; warps 2..5 stage the epilogue inputs,
// read the accumulator out of TMEM (each warp its 32-lane quarter) and, with the
// other two warps, run the same tile finish as the mma.sync path.
constexpr int kTcThreads = 192;

template <int NT>
struct TcCfg {
  static_assert(NT == 64 || NT == 128, "token tiles of 64 or 128 rows (two CTAs per SM)");
  static constexpr int kStages = NT == 128 ? 3 : 4;
  static constexpr int kWBytes = kBN * kBK * 2;
  static constexpr int kXBytes = NT * kBK * 2;
  static constexpr int kStageBytes = kWBytes + kXBytes;
  static constexpr int kPipeBytes = kStages * kStageBytes;
  static constexpr int kTileBytes = NT * kTilePad * 4;
  static_assert(kTileBytes <= kPipeBytes, "epilogue tile reuses the pipeline buffers");
  static constexpr int kTmemCols = NT;  // fp32 accumulator: one column per token row
  // barriers, TMEM address, row scales [NT], weight-row scales [kBN], (position, slot) [NT]
  static constexpr int kSmemBytes = kPipeBytes + (2 * kStages + 1) * 8 + 16 + 16 + NT * 4 + kBN * 4 + NT * 8 + 1024;
};

// Epilogue inputs that do not depend on the accumulator, placed in shared memory
// by the four TMEM warps (t = 0..127) while the MMAs run: the weight-row scales
// of the tile's columns, the row scale of each row this split finishes (sum of
// the previous kernel's per-tile r^2, in the same order as the epilogue would)
// and, for QKV, each row's position and KV slot.
template <int EPI>
SPEC_DEVICE_INLINE void tc_prep(const EpiParams& p, int m0, int n0, float* s_scale, float* s_rs, int2* s_ps, int t,
                                int w, int lane, int r_lo, int r_hi) {
  s_rs[t] = __ldg(p.rscale + n0 + t);
  for (int r0 = r_lo + w; r0 < r_hi; r0 += 8 * 4) {  // eight rows per warp at a time
    float ss[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = r0 + j * 4;
      float a = 0.f;
      if (r < r_hi && p.ssq_in)
        for (int tt = lane; tt < p.ssq_tiles; tt += 32) a += __ldcg(p.ssq_in + (long long)tt * p.ssq_stride + m0 + r);
      ss[j] = a;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = r0 + j * 4;
      const float sum = warp_sum(ss[j]);
      if (r < r_hi && lane == 0) s_scale[r] = p.ssq_in ? rsqrtf(sum * p.inv_d + p.eps) : 1.f;
    }
  }
  // The epilogue's other inputs are read from memory once the accumulator is
  // ready; by then the weight stream (and, before O, the KV cache) has usually
  // pushed them out of L2, so they are brought back into L2 now: each row's RoPE
  // angles (QKV tiles of rotated heads) or residual segment (O and down).
  if constexpr (EPI == kEpiQKV) {
    const bool rotated = n0 / p.hd < p.Hq + p.Hkv;
    for (int r = r_lo + t; r < r_hi; r += 128) {
      const int pos = __ldcg(p.row_pos + m0 + r);
      s_ps[r] = make_int2(pos, __ldcg(p.row_slot + m0 + r));
      if (rotated) {
        l2_prefetch_bulk(p.rope_cos + (long long)pos * (p.hd >> 1), (uint32_t)p.hd * 2);
        l2_prefetch_bulk(p.rope_sin + (long long)pos * (p.hd >> 1), (uint32_t)p.hd * 2);
      }
    }
  }
  if constexpr (EPI == kEpiResid)
    for (int r = r_lo + t; r < r_hi; r += 128) l2_prefetch_bulk(p.resid + (long long)(m0 + r) * p.d + n0, kBN * 4);
}

template <int NT, int EPI>
__global__ void __launch_bounds__(kTcThreads, 2)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ EpiParams p) {
  using C = TcCfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kPipeBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* accum = empty + C::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  // 16-byte aligned: the epilogue reads s_rs as float4
  float* s_scale = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(tmem_slot + 4) + 15) & ~uintptr_t(15));
  float* s_rs = s_scale + NT;
  int2* s_ps = reinterpret_cast<int2*>(s_rs + kBN);
  __shared__ int s_fail;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.z * kBN;
  const int split = blockIdx.y;
  const int m0 = blockIdx.x * NT;
  const int n_act = min(NT, (p.M - m0 + 15) & ~15);  // token rows the MMAs cover
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
      if (!p.late_dependents) pdl_launch_dependents();
      for (int kb = 0; kb < pre; ++kb) tma_load_2d(stage_x(kb), &tmX, (kb0 + kb) * kBK, m0, &full[kb]);
      for (int kb = pre; kb < nkb; ++kb) {
        const int s = kb % C::kStages;
        const uint32_t use = kb / C::kStages;
        if (!mbar_wait(&empty[s], (use - 1) & 1, p.status)) break;
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
        tma_load_2d_hint(stage_w(s), &tmW, (kb0 + kb) * kBK, n0, &full[s], pol);
        tma_load_2d(stage_x(s), &tmX, (kb0 + kb) * kBK, m0, &full[s]);
      }
      l2_prefetch_share(p.l2_next, p.l2_next_bytes);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------- MMA issue (1 thread)
    if (lane == 0) {
      // MMA width: the tile's token rows rounded up to 16 (a ragged last tile
      // multiplies only its own rows)
      const uint32_t idesc = idesc_f16_f32(kBN, n_act);
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
    if (!p.late_dependents) pdl_launch_dependents();
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int nl = q * 32 + lane;      // weight row of this thread within the tile
    int r_lo, r_hi;
    tile_rows<NT>(p, m0, r_lo, r_hi);
    tc_prep<EPI>(p, m0, n0, s_scale, s_rs, s_ps, threadIdx.x - 64, warp - 2, lane, r_lo, r_hi);
    const bool done = mbar_wait(accum, 0, p.status);
    tc_fence_after();
    if (!done) s_fail = 1;
    float* tile = reinterpret_cast<float*>(smem);  // MMAs and loads are done with the stages
    if (done) {
#pragma unroll 1
      for (int c0 = 0; c0 < n_act; c0 += 16) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) tile[(c0 + i) * kTilePad + nl] = v[i];
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
  if (s_fail) {
    if (p.splits > 1) {  // still take part in the cluster barriers
      cluster_arrive();
      cluster_wait();
      cluster_arrive();
      cluster_wait();
    }
    return;
  }
  if (warp < 2) pdl_wait();  // outputs are written below by every warp
  EpiPre<EPI, kTcThreads, NT> pre;  // loads its epilogue inputs row by row
  finish_tile<EPI, kTcThreads, NT, true, 8>(p, pre, reinterpret_cast<float*>(smem), s_scale, m0, n0, threadIdx.x,
                                            warp, lane, s_rs, s_ps);
  if (p.late_dependents) pdl_launch_dependents();
  __syncwarp();
  if (p.splits > 1) cluster_wait();  // the other splits are done reading this CTA's tile
}

// ----------------------------------------------------------------------------
// CTA-pair path (tcgen05 cta_group::2) from 65 token rows: two CTAs on two SMs
// share one MMA of 256 weight rows x N token rows (N up to 256).  Each CTA stages
// its own 128 weight rows and half of the tile's token rows per k-block (the pair
// MMA reads A and B from both CTAs' shared memory) and receives 128 lanes x N
// columns of the accumulator in its own tensor memory.  Per SM that is half the
// staged bytes per MMA of a single-CTA tile with the same token rows, and one
// weight slab serves up to 256 token rows (one pass over the weights up to 256
// rows, where 128-row single-CTA tiles read each slab twice).
//   * Warp 0 of each CTA drives TMA into its own stages; the loads complete on
//     the even CTA's barrier, which expects both CTAs' bytes.
//   * One thread of the even CTA issues the pair MMAs and commits each stage to
//     the empty barriers of both CTAs (multicast), and the accumulator likewise.
//   * Warps 2..5 of each CTA stage the epilogue inputs, then read their CTA's
//     accumulator out of tensor memory in chunks of at most 192 token rows and,
//     with the other two warps, run the common tile finish on each chunk (the
//     fp32 chunk, rows x 132 x 4 bytes, reuses the pipeline buffers).
// Split-K runs as a cluster of (2, S, 1) CTAs: the pair of split j holds cluster
// ranks 2j and 2j + 1.  Two CTAs per SM.
// Tensor memory: a pair allocates the same columns on both of its SMs.  With the
// pair on the two SMs of one TPC, both SMs hold the same CTAs' allocations, so a
// pair never waits for columns that are free on one SM only (a wait that a CTA
// holding columns on the other SM, itself waiting at a cluster barrier for this
// pair, could never end).  Each pair checks its placement before it allocates
// and, placed otherwise, computes nothing and reports SPEC_ERR_UNSUPPORTED.
constexpr int kTc2PipeBytes = 104 * 1024;
constexpr int kTc2MaxRows = 256;    // token rows per tile (MMA N)
constexpr int kTc2ChunkRows = 192;  // token rows per epilogue chunk
constexpr int kTc2MaxStages = 8;
static_assert(kTc2ChunkRows * kTilePad * 4 <= kTc2PipeBytes, "epilogue chunk reuses the pipeline buffers");

struct Tc2Cfg {
  // barriers, TMEM address, row scales [rows], weight-row scales [kBN], (position, slot) [rows]
  static constexpr int kSmemBytes =
      kTc2PipeBytes + (2 * kTc2MaxStages + 1) * 8 + 16 + 16 + kTc2MaxRows * 4 + kBN * 4 + kTc2MaxRows * 8 + 1024;
};
// two CTAs per SM (228 KB of shared memory per SM, 1 KB reserved per CTA), and no third
static_assert(2 * (Tc2Cfg::kSmemBytes + 1024) <= 228 * 1024 && 3 * (Tc2Cfg::kSmemBytes + 1024) > 228 * 1024,
              "the pair kernel runs two CTAs per SM");

template <int EPI>
__global__ void __launch_bounds__(kTcThreads, 2)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ EpiParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTc2PipeBytes);
  uint64_t* empty = full + kTc2MaxStages;
  uint64_t* accum = empty + kTc2MaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  float* s_scale = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(tmem_slot + 4) + 15) & ~uintptr_t(15));
  float* s_rs = s_scale + kTc2MaxRows;
  int2* s_ps = reinterpret_cast<int2*>(s_rs + kBN);
  __shared__ int s_fail;
  __shared__ uint32_t s_sm;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int pr = blockIdx.x & 1;               // position in the pair: 0 issues the MMAs
  const uint32_t crank = cluster_ctarank();    // pr + 2 * blockIdx.y
  const uint32_t lead = crank & ~1u;
  const int n0 = blockIdx.z * (2 * kBN) + pr * kBN;
  const int m0 = (blockIdx.x >> 1) * p.tok_tile;
  const int rows = min(p.tok_tile, p.M - m0);
  const int n_act = min(p.tok_tile, (rows + 15) & ~15);  // MMA N: the tile's rows rounded up to 16
  const int xbox = p.tok_tile / 2;                      // token rows per CTA and stage (TMA box)
  const int stage_bytes = kBN * kBK * 2 + xbox * kBK * 2;
  const int stages = min(kTc2MaxStages, kTc2PipeBytes / stage_bytes);
  const uint32_t tmem_cols = n_act <= 32 ? 32 : n_act <= 64 ? 64 : n_act <= 128 ? 128 : 256;
  const int ch = p.tok_chunk;                          // epilogue chunk rows (same for every tile)
  const int nch = (p.tok_tile + ch - 1) / ch;
  const int kb0 = blockIdx.y * p.kb_per_split;
  const int nkb = min(p.kb_per_split, p.kb_total - kb0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    s_fail = 0;
    s_sm = sm_id();
    fence_barrier_init();
  }
  __syncwarp();
  // The peer's loads complete on the even CTA's barriers and the even CTA's MMAs
  // commit to both CTAs' barriers: all of them are initialised before either runs.
  cluster_arrive();
  cluster_wait();
  // the pair on the two SMs of one TPC (SM ids 2t, 2t + 1), or nothing at all
  const bool placed = (ld_dsmem_u32(mapa_u32(smem_u32(&s_sm), crank ^ 1u)) ^ sm_id()) == 1u;
  if (!placed && threadIdx.x == 0) {
    s_fail = 1;
    if (pr == 0) set_status(p.status, SPEC_ERR_UNSUPPORTED);
  }
  const int pre = min(nkb, stages);
  const uint64_t pol = l2_policy_evict_first();
  if (placed && threadIdx.x == 0 && nkb > 0) {  // weights never depend on the previous kernel
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    for (int kb = 0; kb < pre; ++kb) {
      if (pr == 0) mbar_arrive_expect_tx(&full[kb], 2 * stage_bytes);
      tma_load_2d_pair_hint(smem + kb * stage_bytes, &tmW, (kb0 + kb) * kBK, n0,
                            mapa_u32(smem_u32(&full[kb]), lead), pol);
    }
  }
  __syncwarp();
  if (warp == 1 && placed) {
    tmem_alloc2(tmem_slot, tmem_cols);
    tmem_relinquish2();
  }
  tc_fence_before();
  cluster_arrive();  // both CTAs of every pair hold their tensor memory
  cluster_wait();
  tc_fence_after();
  const uint32_t tmem = placed ? *tmem_slot : 0u;

  auto stage_w = [&](int s) { return smem + s * stage_bytes; };
  auto stage_x = [&](int s) { return smem + s * stage_bytes + kBN * kBK * 2; };

  if (!placed) {
    // nothing staged, nothing issued: straight to the failure path below
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nkb > 0) {
      const int xrow = m0 + pr * (n_act / 2);  // this CTA's half of the MMA's token rows
      pdl_wait();
      if (!p.late_dependents) pdl_launch_dependents();
      for (int kb = 0; kb < pre; ++kb)
        tma_load_2d_pair(stage_x(kb), &tmX, (kb0 + kb) * kBK, xrow, mapa_u32(smem_u32(&full[kb]), lead));
      for (int kb = pre; kb < nkb; ++kb) {
        const int s = kb % stages;
        const uint32_t use = kb / stages;
        if (!mbar_wait(&empty[s], (use - 1) & 1, p.status)) break;
        const uint32_t bar = mapa_u32(smem_u32(&full[s]), lead);
        if (pr == 0) mbar_arrive_expect_tx(&full[s], 2 * stage_bytes);
        tma_load_2d_pair_hint(stage_w(s), &tmW, (kb0 + kb) * kBK, n0, bar, pol);
        tma_load_2d_pair(stage_x(s), &tmX, (kb0 + kb) * kBK, xrow, bar);
      }
      l2_prefetch_share(p.l2_next, p.l2_next_bytes);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------- pair MMA issue (even CTA, 1 thread)
    if (lane == 0 && pr == 0) {
      const uint32_t idesc = idesc_f16_f32(2 * kBN, n_act);
      const uint16_t both = (uint16_t)(3u << lead);
      int kb = 0;
      for (; kb < nkb; ++kb) {
        const int s = kb % stages;
        const uint32_t use = kb / stages;
        if (!mbar_wait(&full[s], use & 1, p.status)) {
          s_fail = 1;
          break;
        }
        tc_fence_after();
        const uint32_t wb = smem_u32(stage_w(s)), xb = smem_u32(stage_x(s));
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          tc_mma2(tmem, sdesc_k_sw128(wb + kk * 32), sdesc_k_sw128(xb + kk * 32), idesc, (kb | kk) != 0);
        // the stage is free in both CTAs once these MMAs have read it (committed only
        // when a producer will wait for it: nothing arrives after the accumulator)
        if (kb + stages < nkb) tc_commit2_mc(&empty[s], both);
      }
      if (nkb <= 0) s_fail = 1;
      tc_commit2_mc(accum, both);  // arrives in both CTAs when every MMA issued above has completed
    }
    __syncwarp();
  } else {
    // ------------------- epilogue inputs while the MMAs run (warps 2..5), then wait
    pdl_wait();
    if (!p.late_dependents) pdl_launch_dependents();
    for (int c = 0; c < nch; ++c) {  // the rows this split finishes in each chunk
      int lo, hi;
      tile_rows<kTc2ChunkRows>(p, m0 + c * ch, lo, hi, min(ch, p.tok_tile - c * ch));
      tc_prep<EPI>(p, m0, n0, s_scale, s_rs, s_ps, threadIdx.x - 64, warp - 2, lane, c * ch + lo, c * ch + hi);
    }
    const bool done = mbar_wait(accum, 0, p.status);
    tc_fence_after();
    if (!done) s_fail = 1;
  }
  // A failure seen by either CTA of the pair (a bounded wait that ran out) holds
  // for both: the flag is copied into the peer before the cluster barrier below.
  __syncthreads();
  if (threadIdx.x == 0 && s_fail) st_dsmem_u32(mapa_u32(smem_u32(&s_fail), crank ^ 1u), 1u);
  __syncwarp();
  cluster_arrive();
  cluster_wait();
  if (s_fail) {
    for (int c = 0; c < nch; ++c)
      if (p.splits > 1) {  // still take part in the cluster barriers of each chunk
        cluster_arrive();
        cluster_wait();
        cluster_arrive();
        cluster_wait();
      }
    if (warp == 1 && placed) {
      tc_fence_after();
      tmem_dealloc2(tmem, tmem_cols);
    }
    return;
  }
  if (warp < 2) pdl_wait();  // outputs are written below by every warp
  float* tile = reinterpret_cast<float*>(smem);  // the pair's MMAs and this CTA's loads are done
  for (int c = 0; c < nch; ++c) {
    const int c0 = c * ch;
    if (warp >= 2) {
      const int q = warp & 3;        // TMEM lane quarter this warp may access
      const int nl = q * 32 + lane;  // weight row of this thread within the CTA's 128
      const int c1 = min(n_act, c0 + ch);
#pragma unroll 1
      for (int col = c0; col < c1; col += 16) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + col, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) tile[(col - c0 + i) * kTilePad + nl] = v[i];
      }
      tc_fence_before();
    }
    __syncthreads();
    EpiPre<EPI, kTcThreads, kTc2ChunkRows> pre;  // loads its epilogue inputs row by row
    // rows [c0, c0 + ch) of the token tile, never past its end (or past M)
    finish_tile<EPI, kTcThreads, kTc2ChunkRows, true, 8>(p, pre, tile, s_scale + c0, m0 + c0, n0, threadIdx.x,
                                                         warp, lane, s_rs, s_ps + c0, pr, 2,
                                                         min(ch, p.tok_tile - c0));
    // The tile is reused by the next chunk once every reader is done: the other
    // splits (they arrived after reading it) and this CTA's own epilogue threads.
    __syncwarp();
    if (p.splits > 1) cluster_wait();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem, tmem_cols);
  }
  if (p.late_dependents) pdl_launch_dependents();
}

// Kernel, block size and dynamic shared memory of the projection for a token tile.
template <int BM, int EPI>
struct Kern {
  static constexpr bool kTc = BM >= 64;  // tcgen05 tiles of 64 / 128 token rows (chosen from 17 rows)
  static auto fn() {
    if constexpr (kTc) {
      return gemm_tc_kernel<BM, EPI>;
    } else {
      return gemm_swapab_kernel<BM, EPI>;
    }
  }
  static constexpr int kThreadsPerCta = kTc ? kTcThreads : kThreads;
  static constexpr int kSmem = kTc ? TcCfg<kTc ? BM : 128>::kSmemBytes : GemmCfg<kTc ? 8 : BM>::kSmemBytes;
};

template <int BM, int EPI>
cudaError_t configure() {
  static bool done = false;
  if (done) return cudaSuccess;
  using K = Kern<BM, EPI>;
  cudaError_t e = cudaFuncSetAttribute(K::fn(), cudaFuncAttributeMaxDynamicSharedMemorySize, K::kSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(K::fn(), cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) done = true;
  return e;
}

// Split-K runs each tile's splits as one cluster of (1, splits, 1) CTAs.
template <int BM, int EPI>
cudaError_t launch_proj(const CUtensorMap* tmW, const CUtensorMap* tmX, EpiParams p, cudaStream_t st) {
  using K = Kern<BM, EPI>;
  if (cudaError_t e = configure<BM, EPI>()) return e;
  // token tiles fastest: the tiles of one weight slab are dispatched side by side,
  // so a slab streamed from HBM for one token tile is still in L2 for the next
  dim3 grid((p.M + BM - 1) / BM, p.splits, p.N / kBN);
  // two CTAs per SM: a grid beyond that is more than one wave (measured at 320 rows:
  // the gate/up projection's 672 CTAs releasing the down projection early left part
  // of down's clusters for a second wave, +25 us per layer)
  p.late_dependents = (long long)grid.x * grid.y * grid.z > 2LL * p.sm_count ? 1 : 0;
  if (p.splits == 1) return launch_k(K::fn(), grid, dim3(K::kThreadsPerCta), K::kSmem, st, *tmW, *tmX, p);
  return launch_k_cluster(K::fn(), grid, dim3(K::kThreadsPerCta), K::kSmem, st, dim3(1, p.splits, 1), *tmW, *tmX,
                          p);
}

// Pair kernel: (2 x token tiles, splits, N / 256) CTAs in clusters of (2, splits, 1).
template <int EPI>
cudaError_t launch_proj2(const CUtensorMap* tmW, const CUtensorMap* tmX, EpiParams p, cudaStream_t st) {
  static bool done = false;
  if (!done) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc2_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Tc2Cfg::kSmemBytes);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemm_tc2_kernel<EPI>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    done = true;
  }
  const int ntt = (p.M + p.tok_tile - 1) / p.tok_tile;
  dim3 grid(2 * ntt, p.splits, p.N / (2 * kBN));
  p.late_dependents = (long long)grid.x * grid.y * grid.z > 2LL * p.sm_count ? 1 : 0;
  return launch_k_cluster(gemm_tc2_kernel<EPI>, grid, dim3(kTcThreads), Tc2Cfg::kSmemBytes, st,
                          dim3(2, p.splits, 1), *tmW, *tmX, p);
}

// How many (1, s, 1) clusters of the projection kernel fit on the GPU at once.
template <int BM>
int max_active_clusters(int s) {
  static std::mutex mu;
  static int cache[kMaxSplits + 1] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (cache[s] == 0) {
    using K = Kern<BM, kEpiResid>;
    int n = 0;
    if (configure<BM, kEpiResid>() == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(1, s, 1);
      cfg.blockDim = dim3(K::kThreadsPerCta);
      cfg.dynamicSmemBytes = K::kSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 1;
      attr[0].val.clusterDim.y = s;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, K::fn(), &cfg) != cudaSuccess) n = 0;
    }
    (void)cudaGetLastError();
    cache[s] = n > 0 ? n : -1;
  }
  return cache[s];
}

static_assert(TcCfg<64>::kSmemBytes <= GemmCfg<8>::kSmemBytes && TcCfg<128>::kSmemBytes <= GemmCfg<8>::kSmemBytes &&
                  kTcThreads <= kThreads,
              "the mma.sync kernel's footprint bounds the 64/128-row tcgen05 kernel's");


int max_active_clusters_bm(int BM, int s) {
  switch (BM) {
    case 8: return max_active_clusters<8>(s);
    case 16: return max_active_clusters<16>(s);
    // The occupancy calculator reports one CTA per SM for the tcgen05 kernel
    // whatever its footprint (measured), while two of its 64- and 128-row CTAs
    // (~100 KB of shared memory, <= 128 TMEM columns each) do run side by side;
    // the mma.sync kernel's two-per-SM footprint stands in for the cluster count.
    default: return max_active_clusters<8>(s);  // 64 and 128 rows
  }
}

template <int EPI>
cudaError_t launch_epi(const CUtensorMap* tmW, const CUtensorMap* tmX, int BM, const EpiParams& p,
                       cudaStream_t st) {
  switch (BM) {  // up to 16 token rows: mma.sync (HBM-bound); from 17: tcgen05
    case kPairBM: return launch_proj2<EPI>(tmW, tmX, p, st);
    case 8: return launch_proj<8, EPI>(tmW, tmX, p, st);
    case 16: return launch_proj<16, EPI>(tmW, tmX, p, st);
    case 64: return launch_proj<64, EPI>(tmW, tmX, p, st);
    case 128: return launch_proj<128, EPI>(tmW, tmX, p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int choose_bm(int M) {
  // measured on whole rounds: mma.sync up to 16 rows; tcgen05 64-row tiles (MMA
  // width = rows rounded up to 16) from 17 rows, 6-7% faster than mma.sync at
  // 20-30 rows and 8% slower at 16; beyond 128 rows several 128-row tiles (two
  // 128-row CTAs per SM beat one 256-row CTA by 7-11% at 192-320 rows)
  if (M <= 8) return 8;
  if (M <= 16) return 16;
  if (M <= 64) return 64;
  return 128;
}

bool pair_rows(int M) {
  // Measured on whole rounds at the 8B widths (B = 16..64, widths 2..16): the pair
  // kernel is faster from 65 to 192 token rows (one tile), from 257 to 384 (two
  // tiles of up to 192) and beyond 512; at 193..256 and 385..512 rows, where it
  // would run tiles of more than 192 rows (three 32 KB stages per CTA), the
  // single-CTA kernel's 128-row tiles are faster, and below 65 rows too.
  return (M > 64 && M <= 192) || (M > 256 && M <= 384) || M > 512;
}

int pair_tile_rows(int M) {
  // As few token tiles of at most 256 rows as possible -- each is one more pass of
  // the weights through L2 -- unless tiles of at most 192 rows come to a multiple
  // of four: the widest projection (gate/up, 112 weight pairs) then fills its
  // waves of two CTAs per SM (4 tiles: 896 CTAs, 2.95 waves of 304; 3 tiles: 672,
  // 2.2 waves).  Measured: 768 rows 13.4 ms in 4 tiles, 14.7 ms in 3.
  const int n_wide = (M + kTc2MaxRows - 1) / kTc2MaxRows, n_narrow = (M + kTc2ChunkRows - 1) / kTc2ChunkRows;
  const int ntt = (n_narrow % 4 == 0 && n_wide % 4 != 0) ? n_narrow : n_wide;
  int T = ((M + ntt - 1) / ntt + 15) & ~15;
  if (T > kTc2ChunkRows) T = (T + 31) & ~31;  // two epilogue chunks of a multiple of 16 rows
  return T;
}

int choose_splits(int N, int K, int M, int BM, int sm_count, int max_splits) {
  if (BM == kPairBM) {
    // The most splits for which every tile's cluster of 2 x splits CTAs is resident
    // in one wave (two CTAs per SM), with every split non-empty and at least 4
    // k-blocks long.
    const int T = pair_tile_rows(M);
    const int pairs = (N / (2 * kBN)) * ((M + T - 1) / T);
    const int kb = K / kBK;
    const int smax = std::min({max_splits, kMaxSplits / 2, std::max(1, kb / 4), std::max(1, sm_count / pairs)});
    for (int s = smax; s > 1; --s) {
      const int per = (kb + s - 1) / s;
      if ((kb + per - 1) / per != s) continue;  // some split would be empty
      if (pairs <= max_active_clusters_bm(8, 2 * s)) return s;
    }
    return 1;
  }
  // The most splits (cluster size) for which every tile's cluster is resident in
  // one wave (two CTAs per SM for every token tile; the GPC layout limits how
  // many clusters fit), with every split non-empty and at least 4 k-blocks long.
  const int tiles = (N / kBN) * ((M + BM - 1) / BM);
  const int kb = K / kBK;
  const int slots = (BM <= 128 ? 2 : 1) * sm_count;
  const int smax = std::min({max_splits, kMaxSplits, std::max(1, kb / 4), std::max(1, slots / tiles)});
  for (int s = smax; s > 1; --s) {
    const int per = (kb + s - 1) / s;
    if ((kb + per - 1) / per != s) continue;  // some split would be empty
    if (tiles <= max_active_clusters_bm(BM, s)) return s;
  }
  return 1;
}

cudaError_t launch_gemm_epi(int epi, const CUtensorMap* tmW, const CUtensorMap* tmX, int BM, EpiParams p,
                            cudaStream_t st) {
  p.kb_total = p.K / kBK;
  p.tok_tile = BM == kPairBM ? pair_tile_rows(p.M) : 0;
  p.tok_chunk = p.tok_tile > kTc2ChunkRows ? p.tok_tile / 2 : p.tok_tile;
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
