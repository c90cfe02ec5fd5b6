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
// K/V pages (64 tokens x head_dim fp16 per kv head) are streamed by TMA with
// the 128-byte swizzle into a 3-stage mbarrier pipeline fed by one producer
// warp.  Consumer warps are (row tile, key group) pairs: a warp owns 16 query
// rows and 64/KG keys of every page and runs QK^T and PV on mma.sync with an
// online softmax in fp32 (exp2 domain).  Splitting the keys of a page over KG
// warps puts a warp on every scheduler, so the short dependent MMA chains of a
// 16-row tile overlap instead of running back to back.  A sequence's pages are
// split over a thread-block cluster of 1 to 16 CTAs (the widest whose grid fits
// one wave); every warp leaves its partial (unnormalised O, running max, running
// sum) in its CTA's shared memory and the cluster merges all CS x KG partials of
// a row through distributed shared memory with log-sum-exp weights, so the
// partials never go to HBM and no separate merge launch is needed.
#include <cooperative_groups.h>
#include <math.h>

#include "common.cuh"
#include "launch.cuh"

namespace cg = cooperative_groups;

namespace spec {

namespace {

// 2^x on the special-function unit (PTX ex2.approx, relative error about 2^-22;
// subnormal results flush to zero).  The scores it exponentiates are rounded to
// fp16 for the PV product, so the approximation is far below that rounding.
SPEC_DEVICE_INLINE float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr int kAttnStages = 3;
constexpr int kMaxRowTiles = 4;       // up to 64 query rows (W * group) per CTA
constexpr int kMaxConsumerWarps = 8;  // row tiles x key groups
constexpr int kMaxKgSlots = 6;        // partials of key groups > 0 (row tiles x (KG - 1))

// Key groups per page for a launch with `row_tiles` row tiles: four consumer warps
// at most, so a CTA stays small enough for several to share an SM.  Splitting keys
// pays off only when a CTA has pages enough to amortise the extra partials in the
// merge (measured on GB300: from about 4 pages per CTA with one row tile, 8 with
// two; a four-way split at 2 pages and a two-way one at 2-3 pages were slower or
// within noise).
inline int key_groups(int row_tiles, int pages_per_cta) {
  if (row_tiles == 1 && pages_per_cta >= 4) return 4;
  if (row_tiles == 2 && pages_per_cta >= 8) return 2;
  return 1;
}

template <int HD>
struct AttnCfg {
  static constexpr int kHalves = HD / 64;
  static constexpr int kTileBytes = kPage * HD * 2;  // one K (or V) page of one kv head
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kSmemBytes = kAttnStages * kStageBytes + 2 * kAttnStages * 8 + 1024;
};

template <int HD, int CS, int KG>
__global__ void __launch_bounds__((kMaxConsumerWarps + 1) * 32)
    attention_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ AttnParams p) {
  using C = AttnCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kAttnStages * C::kStageBytes);
  uint64_t* empty = full + kAttnStages;
  __shared__ int s_fail;
  // ancestor masks in shared memory: read with a per-row index, which from the
  // parameter bank would be a divergent constant load repeated for every page
  __shared__ uint32_t s_anc[16];
  cg::cluster_group cluster = cg::this_cluster();

  const int rank = (int)cluster.block_rank();  // == blockIdx.x: the split of this CTA
  const int kvh = blockIdx.y;
  const int b = p.seq_order ? p.seq_order[blockIdx.z] : blockIdx.z;  // longest cache first
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_cons = blockDim.x / 32 - 1;  // consumer warps: (row tile, key group) pairs
  const int grp = p.Hq / p.Hkv;
  constexpr int KT = 4 / KG;                // 16-key tiles of a page per consumer warp

  // Sequence state and the cached pages were written by kernels that completed
  // before the QKV projection (this kernel's predecessor) passed its own
  // griddepcontrol.wait, which it does before letting this kernel launch; only
  // q and the window's K/V come from the predecessor itself.  The successor (the
  // O projection) only prefetches weights before its own wait, so it may launch
  // right away -- or, for short attentions (p.late_trigger), once this CTA's
  // queries have arrived: its weight stream would otherwise queue ahead of them.
  if (!p.late_trigger) pdl_launch_dependents();
  const int sid = p.seq_ids[b];
  const bool sid_ok = sid >= 0 && sid < p.max_batch;  // a bad id was flagged by the prepare kernel
  const int L = p.seq_start[b];
  const int Wb = p.seq_wlen[b];      // this sequence's window rows (<= p.W)
  const int row0 = p.seq_rowoff[b];  // its first flat row
  const int rows = Wb * grp;
  const int n_keys = L + Wb;
  const int n_pages = sid_ok ? min((n_keys + kPage - 1) / kPage, p.max_pages) : 0;
  const int pps = (n_pages + CS - 1) / CS;
  const int pg0 = rank * pps;
  const int pg1 = min(pg0 + pps, n_pages);
  const int npg = max(0, pg1 - pg0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAttnStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], n_cons);
    }
    s_fail = 0;
    fence_barrier_init();
  }
  if (threadIdx.x < 16) s_anc[threadIdx.x] = p.anc[threadIdx.x];
  __syncthreads();

  // partials of this CTA, reusing the stage buffers once the pipeline is drained
  float* part_o = reinterpret_cast<float*>(smem);            // [rows][HD]
  float* part_m = part_o + kMaxRowTiles * 16 * HD;           // [rows]
  float* part_l = part_m + kMaxRowTiles * 16;                // [rows]
  float* kg_o = part_l + kMaxRowTiles * 16;                  // [slots][16][HD] key-group partials
  float* kg_m = kg_o + kMaxKgSlots * 16 * HD;                // [slots][16]
  float* kg_l = kg_m + kMaxKgSlots * 16;
  static_assert((kMaxRowTiles * 16 * (HD + 2) + kMaxKgSlots * 16 * (HD + 2)) * 4 <=
                    kAttnStages * 2 * kPage * HD * 2,
                "partials fit in the stage buffers");

  if (warp == n_cons) {
    // --------------------------------------------------------------- producer
    if (lane == 0 && npg > 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int32_t* pt = p.page_table + (long long)sid * p.max_pages;
      bool waited = false;
      for (int i = 0; i < npg; ++i) {
        const int s = i % kAttnStages;
        const uint32_t use = i / kAttnStages;
        if (!waited && (pg0 + i + 1) * kPage > L) {  // this page holds window slots
          pdl_wait();
          waited = true;
        }
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
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- consumers
    pdl_wait();  // q is written by the QKV projection
    // the successor may launch, and the next weights go to L2: at once, or (late
    // trigger) after this warp's first use of its queries
    auto release_successor = [&] {
      if (warp == 0 && lane == 0) {
        if (p.late_trigger) pdl_launch_dependents();
        l2_prefetch_share(p.l2_next[0], p.l2_next_bytes[0]);
        l2_prefetch_share(p.l2_next[1], p.l2_next_bytes[1]);
      }
    };
    if (!p.late_trigger) release_successor();
    const int g = lane >> 2, c = lane & 3;
    const int rt = warp / KG, kg = warp % KG;  // row tile, key group (keys kg*16*KT .. of each page)
    // query rows of this thread: r0 = rt*16 + g, r1 = r0 + 8; row r -> window row j = r / grp
    int jrow[2], head[2];
    bool valid[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = rt * 16 + g + 8 * h;
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
        const act_t* qr =
            p.q + ((long long)(row0 + jrow[h]) * p.Hq + head[h]) * HD + ks * 16 + 2 * c;
        const uint32_t lo = valid[h] ? *reinterpret_cast<const uint32_t*>(qr) : 0u;
        const uint32_t hi = valid[h] ? *reinterpret_cast<const uint32_t*>(qr + 8) : 0u;
        qa[ks][h] = lo;       // a0a1 (row g) / a2a3 (row g+8)
        qa[ks][2 + h] = hi;   // a4a5 / a6a7
      }
    }
    const uint32_t anc0 = valid[0] ? s_anc[jrow[0]] : 0u;
    const uint32_t anc1 = valid[1] ? s_anc[jrow[1]] : 0u;
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)HD);

    float acc[HD / 8][4];
#pragma unroll
    for (int t = 0; t < HD / 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY};
    float lrow[2] = {0.f, 0.f};

    for (int i = 0; i < npg; ++i) {
      const int s = i % kAttnStages;
      const uint32_t use = i / kAttnStages;
      if (!mbar_wait(&full[s], use & 1, p.status)) {
        s_fail = 1;
        break;
      }
      const uint32_t kbase = smem_u32(smem + s * C::kStageBytes);
      const uint32_t vbase = kbase + C::kTileBytes;

      // S = Q K^T for this warp's 16*KT keys of the page: 2*KT key tiles of 8
      float sc[2 * KT][4];
#pragma unroll
      for (int t = 0; t < 2 * KT; ++t) sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
        for (int tp = 0; tp < KT; ++tp) {
          const int key = (kg * KT + tp) * 16 + (lane & 7) + ((lane >> 4) & 1) * 8;
          const int d = ks * 16 + ((lane >> 3) & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + (d >> 6) * (kPage * 128) + swz128(key, d & 63), b0, b1, b2, b3);
          mma_f16_16816(sc[2 * tp], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          mma_f16_16816(sc[2 * tp + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
      }
      if (p.late_trigger && i == 0) release_successor();
      // mask + online softmax (exp2 domain)
      float mx[2] = {-INFINITY, -INFINITY};
      // visibility of the page's 64 keys for this thread's two rows (bit k: key
      // key0p + k), then of this thread's keys of the slice (bit t*2 + (e&1))
      uint32_t vb[2];
      {
        const int key0p = (pg0 + i) * kPage;
        const int hist = min(max(L - key0p, 0), kPage);  // cached keys at the page start
        const uint64_t hmask = hist == kPage ? ~0ull : ((1ull << hist) - 1ull);
        const int sh = kg * KT * 16 + 2 * c;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // window rows visible to this row (slots below the sequence's Wb only)
          const uint64_t anc = (h ? anc1 : anc0) & ((1u << Wb) - 1u);
          // window slot w sits at page key L + w - key0p
          const int off = L - key0p;
          uint64_t wmask = 0;
          if (off >= 0 && off < kPage) wmask = anc << off;
          else if (off < 0 && off > -32) wmask = anc >> (-off);
          const uint64_t m = valid[h] ? (hmask | wmask) >> sh : 0ull;
          uint32_t bits = 0;
#pragma unroll
          for (int t = 0; t < 2 * KT; ++t)
            bits |= (uint32_t)((m >> (t * 8)) & 3ull) << (2 * t);
          vb[h] = bits;
        }
      }
#pragma unroll
      for (int t = 0; t < 2 * KT; ++t) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = e >> 1;
          const float v = ((vb[h] >> (t * 2 + (e & 1))) & 1u) ? sc[t][e] * scale_log2 : -INFINITY;
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
        alpha[h] = (mrow[h] == -INFINITY) ? 0.f : fast_exp2(mrow[h] - mnew);
        mrow[h] = mnew;
      }
      float rs[2] = {0.f, 0.f};
#pragma unroll
      for (int t = 0; t < 2 * KT; ++t) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = e >> 1;
          const float pv = (mrow[h] == -INFINITY) ? 0.f : fast_exp2(sc[t][e] - mrow[h]);
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
      // O += P V: P from the score registers (fp16), V via transposed ldmatrix
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        const uint32_t a0 = pack_f16x2(sc[2 * kk][0], sc[2 * kk][1]);
        const uint32_t a1 = pack_f16x2(sc[2 * kk][2], sc[2 * kk][3]);
        const uint32_t a2 = pack_f16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        const uint32_t a3 = pack_f16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < HD / 16; ++dp) {
          const int key = (kg * KT + kk) * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int d = dp * 16 + ((lane >> 4) & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_trans(vbase + (d >> 6) * (kPage * 128) + swz128(key, d & 63), b0, b1, b2, b3);
          mma_f16_16816(acc[2 * dp], a0, a1, a2, a3, b0, b1);
          mma_f16_16816(acc[2 * dp + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      // The stage is refilled by TMA (async proxy) after this arrive: order this
      // thread's ldmatrix reads (generic proxy) of it before that write.
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (p.late_trigger && npg == 0) release_successor();
    // drained: every issued page was consumed, so the stage buffers are free
    // once all consumer warps are here (named barrier over the consumers)
    asm volatile("bar.sync 1, %0;" ::"r"(n_cons * 32) : "memory");
    // key group 0 writes straight into the CTA partial, the others into slots
    const int slot = rt * (KG - 1) + kg - 1;
    float* o_dst = kg == 0 ? part_o : kg_o + slot * 16 * HD - rt * 16 * HD;
    float* m_dst = kg == 0 ? part_m : kg_m + slot * 16 - rt * 16;
    float* l_dst = kg == 0 ? part_l : kg_l + slot * 16 - rt * 16;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = rt * 16 + g + 8 * h;
#pragma unroll
      for (int t = 0; t < HD / 8; ++t) {
        o_dst[r * HD + t * 8 + 2 * c] = acc[t][2 * h];
        o_dst[r * HD + t * 8 + 2 * c + 1] = acc[t][2 * h + 1];
      }
      if (c == 0) {
        m_dst[r] = valid[h] ? mrow[h] : -INFINITY;
        l_dst[r] = valid[h] ? lrow[h] : 0.f;
      }
    }
  }
  // every CTA of the cluster has its partials in shared memory
  if (warp == n_cons) pdl_wait();  // every thread below may write the output
  cluster.sync();
  if (!s_fail) {
    // CTA `rank` merges rows rank, rank + CS, ...: each thread owns 4 consecutive
    // output elements of one row.  The row's partials are the CS CTAs' key-group
    // partials (KG per CTA); they are taken 16 at a time, and each batch's remote
    // loads -- (m, l) and the 4 partial outputs of every partial -- are all issued
    // before any is used, so the merge costs one distributed-shared-memory round
    // trip per batch.  Across batches the running sums are rescaled to the new max.
    // out = sum_p 2^(m_p - max m) o_p / sum_p 2^(m_p - max m) l_p
    constexpr int V4 = HD / 4;
    constexpr int NP = CS * KG;                  // partials per row
    constexpr int NB = NP < 16 ? NP : 16;        // partials per batch
    const int n_my_rows = rows > rank ? (rows - rank + CS - 1) / CS : 0;
    const uint32_t o_base = smem_u32(part_o), m_base = smem_u32(part_m), l_base = smem_u32(part_l);
    const uint32_t ko_base = smem_u32(kg_o), km_base = smem_u32(kg_m), kl_base = smem_u32(kg_l);
    for (int it = threadIdx.x; it < n_my_rows * V4; it += blockDim.x) {
      const int lr = it / V4, d4 = it % V4;
      const int r = rank + lr * CS;
      const int rtr = r / 16, rr = r % 16;
      float mrun = -INFINITY, den = 0.f, n0 = 0.f, n1 = 0.f, n2 = 0.f, n3 = 0.f;
#pragma unroll
      for (int p0 = 0; p0 < NP; p0 += NB) {
        float ms[NB], ls[NB];
        float4 os[NB];
#pragma unroll
        for (int q = 0; q < NB; ++q) {
          const int pi = p0 + q, s_ = pi / KG, k = pi % KG;  // partial pi: CTA s_, key group k
          uint32_t ma, la, oa;
          if (k == 0) {
            ma = m_base + r * 4;
            la = l_base + r * 4;
            oa = o_base + (r * HD + d4 * 4) * 4;
          } else {
            const int sl = (rtr * (KG - 1) + k - 1) * 16 + rr;
            ma = km_base + sl * 4;
            la = kl_base + sl * 4;
            oa = ko_base + (sl * HD + d4 * 4) * 4;
          }
          ms[q] = ld_dsmem_f32(mapa_u32(ma, s_));
          ls[q] = ld_dsmem_f32(mapa_u32(la, s_));
          os[q] = ld_dsmem_f4(mapa_u32(oa, s_));
        }
        float mb = mrun;
#pragma unroll
        for (int q = 0; q < NB; ++q) mb = fmaxf(mb, ms[q]);
        if (mb != -INFINITY && mrun != mb) {  // rescale the running sums to the new max
          const float a = mrun == -INFINITY ? 0.f : fast_exp2(mrun - mb);
          den *= a;
          n0 *= a;
          n1 *= a;
          n2 *= a;
          n3 *= a;
        }
        mrun = mb;
#pragma unroll
        for (int q = 0; q < NB; ++q) {
          const float w = (mb == -INFINITY || ms[q] == -INFINITY) ? 0.f : fast_exp2(ms[q] - mb);
          den += w * ls[q];
          n0 += w * os[q].x;
          n1 += w * os[q].y;
          n2 += w * os[q].z;
          n3 += w * os[q].w;
        }
      }
      const float inv = den > 0.f ? 1.f / den : 0.f;
      const int j = r / grp, hq = kvh * grp + r % grp;
      *reinterpret_cast<uint2*>(p.out + ((long long)(row0 + j) * p.Hq + hq) * HD + d4 * 4) =
          pack_act4(n0 * inv, n1 * inv, n2 * inv, n3 * inv);
    }
  }
  // keep this CTA's shared memory alive until every CTA has read it
  cluster.sync();
}

template <int HD, int CS, int KG>
cudaError_t launch_attention_kg(const CUtensorMap* tmK, const CUtensorMap* tmV, const AttnParams& p, int row_tiles,
                                cudaStream_t st) {
  using C = AttnCfg<HD>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attention_kernel<HD, CS, KG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e == cudaSuccess && CS > 8)
      e = cudaFuncSetAttribute(attention_kernel<HD, CS, KG>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(CS, p.Hkv, p.B);
  return launch_k_cluster(attention_kernel<HD, CS, KG>, grid, dim3((row_tiles * KG + 1) * 32), C::kSmemBytes, st,
                          dim3(CS, 1, 1), *tmK, *tmV, p);
}

template <int HD, int CS>
cudaError_t launch_attention_hd(const CUtensorMap* tmK, const CUtensorMap* tmV, const AttnParams& p,
                                cudaStream_t st) {
  const int rows = p.W * (p.Hq / p.Hkv);
  const int row_tiles = (rows + 15) / 16;
  if (row_tiles > kMaxRowTiles) return cudaErrorInvalidValue;
  const int pages_per_cta = ((p.kv_len_hint + kPage - 1) / kPage + CS - 1) / CS;
  AttnParams q = p;
  q.late_trigger = pages_per_cta <= 2;  // measured: earlier successor launch wins from 3 pages per CTA
  switch (key_groups(row_tiles, pages_per_cta)) {
    case 4: return launch_attention_kg<HD, CS, 4>(tmK, tmV, q, row_tiles, st);
    case 2: return launch_attention_kg<HD, CS, 2>(tmK, tmV, q, row_tiles, st);
    default: return launch_attention_kg<HD, CS, 1>(tmK, tmV, q, row_tiles, st);
  }
}

}  // namespace

cudaError_t launch_attention(const CUtensorMap* tmK, const CUtensorMap* tmV, const AttnParams& p, cudaStream_t st) {
  // The widest cluster (16, 8, 4, 2 or 1 CTAs per sequence and kv head) whose grid
  // fits one CTA per SM while clusters of 8 still do, else the widest that fits two
  // per SM.  Few sequences spread their pages over many SMs, many keep more pages
  // per CTA (and fewer merges).  Measured per round: an 8-CTA cluster alone on its
  // SMs beats a 16-CTA one doubled up at B = 2 (8 kv heads) by 7% at 1K cached
  // tokens and 10% at 4K; from B = 3 doubling up wins at 4K tokens by 6-11% (B = 3,
  // B = 4, 15-node trees) and ties at 1K.
  const int per_sm = p.B * p.Hkv * 8 <= p.sm_count ? 1 : 2;
  int cs = 16;
  while (cs > 1 && p.B * p.Hkv * cs > per_sm * p.sm_count) cs >>= 1;
  if (p.hd == 128) {
    switch (cs) {
      case 16: return launch_attention_hd<128, 16>(tmK, tmV, p, st);
      case 8: return launch_attention_hd<128, 8>(tmK, tmV, p, st);
      case 4: return launch_attention_hd<128, 4>(tmK, tmV, p, st);
      case 2: return launch_attention_hd<128, 2>(tmK, tmV, p, st);
      default: return launch_attention_hd<128, 1>(tmK, tmV, p, st);
    }
  }
  if (p.hd == 64) {
    switch (cs) {
      case 16: return launch_attention_hd<64, 16>(tmK, tmV, p, st);
      case 8: return launch_attention_hd<64, 8>(tmK, tmV, p, st);
      case 4: return launch_attention_hd<64, 4>(tmK, tmV, p, st);
      case 2: return launch_attention_hd<64, 2>(tmK, tmV, p, st);
      default: return launch_attention_hd<64, 1>(tmK, tmV, p, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace spec
