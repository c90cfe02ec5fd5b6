// Top-k / top-p selection of one probability row per thread-block cluster.
//
// Lecture 6 "Optimizing Autoregressive Decode" section 7.3 (top-k keeps the k
// most probable tokens, top-p the smallest top-ranked set that reaches mass p;
// speculative sampling on p and q adjusted alike follows the adjusted p) and
// "Per-step cost versus accepted tokens", section "Reefs" (the renormalisation
// runs at verify time whenever top_k > 1 or top_p < 1).  Readings: rank order is
// p descending with the lower token index first among equal p; top-k is applied
// first and top-p acts on the top-k renormalised distribution; masses are
// R_v = floor(p_v * 2^40), so every set decision is integer arithmetic and does
// not depend on the summation order.
//
// The row is split across the cluster's CTAs (a contiguous vocabulary slice
// each, its probability keys held in shared memory).  Each threshold is found by
// a most-significant-digit-first radix select over the 32-bit keys, 8 bits per
// pass: every CTA builds a 256-bin histogram of counts and masses of its slice
// with 32-bit shared-memory atomics (a mass, at most 2^40, is added as three
// 32-bit parts that cannot overflow for a slice of probabilities; each thread
// first sums runs of equal digits in registers, and a warp whose lanes end on the
// same digit adds once), the histograms are added through distributed shared
// memory, and the bin where the running
// count (top-k) or mass (top-p) from the top reaches the target fixes the next
// 8 bits.  Equal keys at the final threshold are kept in index order: the CTA
// holding the cut finds it with an ordered ballot scan and broadcasts it.
#include <cooperative_groups.h>
#include <math.h>

#include "launch.cuh"
#include "sampling.cuh"

namespace cg = cooperative_groups;

namespace spec {

namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBins = 256;

// A mass R <= 2^40 is accumulated as R[0:12) + R[12:26) << 12 + R[26:) << 26 in three
// 32-bit counters: over at most 2^14 elements (a slice of a row) each part sums to
// less than 2^28, and the native 32-bit shared atomics stay fast under conflicts.
struct SelShared {
  unsigned int cnt[2][kBins];          // this CTA's histogram (double-buffered across passes)
  unsigned int m0[2][kBins], m1[2][kBins], m2[2][kBins];
  unsigned int gc[kBins];              // cluster-wide histogram of the current pass
  unsigned long long gm[kBins];
  unsigned long long red[kSelWarps];
  unsigned long long total;            // this CTA's summed mass (read by the other CTAs)
  unsigned long long all_total;
  unsigned int ties;                   // this CTA's keys equal to the threshold
  unsigned int ties_before;
  int cut;                             // written by the CTA that holds the cut
  int wc[kSelWarps];
  int fail;
  // result of a select
  uint32_t dsel;
  unsigned long long above_c, above_m;
  unsigned int tie_cnt;
  float mx, z;
};

SPEC_DEVICE_INLINE unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

SPEC_DEVICE_INLINE unsigned long long block_sum_u64(unsigned long long v, SelShared& sh) {
  v = warp_sum_u64(v);
  if ((threadIdx.x & 31) == 0) sh.red[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long s = 0;
  for (int w = 0; w < kSelWarps; ++w) s += sh.red[w];
  __syncthreads();
  return s;
}

struct SelectResult {
  uint32_t t;                 // threshold key
  unsigned long long above_c; // keys > t: count
  unsigned long long above_m; //           and mass
  unsigned int tie_cnt;       // keys == t
  bool ok;
};

// Radix select: the largest key t with measure(keys > t) < target <= measure(keys >= t),
// measure = count (by_mass false) or summed 2^-40 mass (by_mass true).
SPEC_DEVICE_INLINE SelectResult radix_select(cg::cluster_group& cluster, SelShared& sh, const uint32_t* keys, int n,
                                             bool by_mass, unsigned long long target, int& pass) {
  const int csize = (int)cluster.num_blocks();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t prefix = 0, mask = 0;
  unsigned long long above_c = 0, above_m = 0;
  unsigned int tie_cnt = 0;
  bool ok = true;
  for (int shift = 24; shift >= 0; shift -= 8) {
    const int buf = (pass++) & 1;
    for (int i = threadIdx.x; i < kBins; i += kSelThreads) {
      sh.cnt[buf][i] = 0;
      sh.m0[buf][i] = sh.m1[buf][i] = sh.m2[buf][i] = 0;
    }
    __syncthreads();
    // The leading digits of a probability row are concentrated in a few bins, so
    // each thread sums a run of equal digits in registers and adds the run when
    // the digit changes; at the end a warp whose lanes hold the same digit adds
    // once.  (Spread digits add element by element.)
    uint32_t cd = 0xffffffffu, cc = 0, c0 = 0, c1 = 0, c2 = 0;
    auto flush = [&](uint32_t dd, uint32_t n_, uint32_t a0, uint32_t a1, uint32_t a2) {
      atomicAdd(&sh.cnt[buf][dd], n_);
      atomicAdd(&sh.m0[buf][dd], a0);
      atomicAdd(&sh.m1[buf][dd], a1);
      atomicAdd(&sh.m2[buf][dd], a2);
    };
    for (int i = threadIdx.x; i < n; i += kSelThreads) {
      const uint32_t key = keys[i];
      if ((key & mask) != prefix) continue;
      const uint32_t d = (key >> shift) & 0xffu;
      const unsigned long long R = key_mass(key);  // <= 2^40
      if (d != cd) {
        if (cc) flush(cd, cc, c0, c1, c2);
        cd = d;
        cc = c0 = c1 = c2 = 0;
      }
      ++cc;
      c0 += (uint32_t)(R & 0xfffu);
      c1 += (uint32_t)((R >> 12) & 0x3fffu);
      c2 += (uint32_t)(R >> 26);
    }
    const uint32_t cd0 = __shfl_sync(0xffffffffu, cd, 0);
    if (__all_sync(0xffffffffu, cd == cd0)) {
      cc = __reduce_add_sync(0xffffffffu, cc);
      c0 = __reduce_add_sync(0xffffffffu, c0);
      c1 = __reduce_add_sync(0xffffffffu, c1);
      c2 = __reduce_add_sync(0xffffffffu, c2);
      if (lane == 0 && cc) flush(cd0, cc, c0, c1, c2);
    } else if (cc) {
      flush(cd, cc, c0, c1, c2);
    }
    __syncthreads();
    cluster.sync();
    for (int bin = threadIdx.x; bin < kBins; bin += kSelThreads) {
      unsigned int c = 0;
      unsigned long long m = 0;
      for (int r = 0; r < csize; ++r) {
        const SelShared* rs = cluster.map_shared_rank(&sh, r);
        c += rs->cnt[buf][bin];
        m += (unsigned long long)rs->m0[buf][bin] + ((unsigned long long)rs->m1[buf][bin] << 12) +
             ((unsigned long long)rs->m2[buf][bin] << 26);
      }
      sh.gc[bin] = c;
      sh.gm[bin] = m;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 255 - 8l down to 248 - 8l: lane order is descending key order
      unsigned long long v[8], s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int bin = 255 - 8 * lane - j;
        v[j] = by_mass ? sh.gm[bin] : (unsigned long long)sh.gc[bin];
        s += v[j];
      }
      unsigned long long inc = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      const unsigned long long base = by_mass ? above_m : above_c;
      const uint32_t reach = __ballot_sync(0xffffffffu, base + inc >= target);
      const int first = reach ? __ffs(reach) - 1 : 31;
      int dloc = 7;
      if (lane == first) {
        unsigned long long run = base + inc - s;
        for (int j = 0; j < 8; ++j) {
          if (run + v[j] >= target) {
            dloc = j;
            break;
          }
          run += v[j];
        }
      }
      const int dstar = 255 - 8 * first - __shfl_sync(0xffffffffu, dloc, first);
      unsigned long long ac = 0, am = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int bin = 255 - 8 * lane - j;
        if (bin > dstar) {
          ac += sh.gc[bin];
          am += sh.gm[bin];
        }
      }
      ac = warp_sum_u64(ac);
      am = warp_sum_u64(am);
      if (lane == 0) {
        sh.dsel = (uint32_t)dstar;
        sh.above_c = ac;
        sh.above_m = am;
        sh.tie_cnt = sh.gc[dstar];
        sh.fail = reach == 0u;
      }
    }
    __syncthreads();
    prefix |= sh.dsel << shift;
    mask |= 0xffu << shift;
    above_c += sh.above_c;
    above_m += sh.above_m;
    tie_cnt = sh.tie_cnt;
    ok = ok && !sh.fail;
    __syncthreads();  // the decision words are rewritten by the next pass
  }
  return SelectResult{prefix, above_c, above_m, tie_cnt, ok};
}

template <PSource SRC>
__global__ void __launch_bounds__(kSelThreads) select_kernel(const __grid_constant__ SelectParams p) {
  extern __shared__ uint32_t keys[];
  __shared__ SelShared sh;
  pdl_wait();
  pdl_launch_dependents();
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int csize = (int)cluster.num_blocks();
  const int V = p.V;
  long long row;
  int set;
  if constexpr (SRC == PSource::kProbs) {
    row = blockIdx.y;
    set = (int)(row / p.rows_per_set);
  } else {
    const int b = blockIdx.z, j = blockIdx.y;
    if (j >= p.seq_wlen[b]) return;  // the whole cluster leaves together
    row = p.seq_rowoff[b] + j;
    set = b;
  }
  const int K = p.top_k ? p.top_k[set] : 0;
  const float TP = p.top_p ? p.top_p[set] : 1.f;
  const bool bad = K < 0 || !(TP > 0.f && TP <= 1.f);
  if (bad && rank == 0 && threadIdx.x == 0) set_status(p.status, SPEC_ERR_INVALID_ARG);
  const bool k_on = !bad && K >= 1 && K < V;
  const bool p_on = !bad && TP < 1.f;
  const int slice = (V + csize - 1) / csize;
  const int s0 = min(V, rank * slice), s1 = min(V, s0 + slice), n = s1 - s0;

  float mx = 0.f, z = 1.f;
  if constexpr (SRC == PSource::kLogits) {
    // merge the LM head's per-128-column statistics of this row (warp 0)
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      float m = -INFINITY;
      for (int t = lane; t < p.n_tiles; t += 32) m = fmaxf(m, p.tstat_max[(long long)t * p.tstat_stride + row]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float zz = 0.f;
      for (int t = lane; t < p.n_tiles; t += 32) {
        const float tm = p.tstat_max[(long long)t * p.tstat_stride + row];
        zz += p.tstat_sum[(long long)t * p.tstat_stride + row] * expf((tm - m) * p.inv_temp);
      }
      zz = warp_sum(zz);
      if (lane == 0) {
        sh.mx = m;
        sh.z = zz;
      }
    }
    __syncthreads();
    mx = sh.mx;
    z = sh.z;
    if (rank == 0 && threadIdx.x == 0) {
      p.row_max[row] = mx;
      p.row_z[row] = z;
    }
  }
  const float* src = SRC == PSource::kProbs ? p.p_in + row * V : p.logits + row * V;
  auto base_prob = [&](int v) -> float {
    if constexpr (SRC == PSource::kProbs) {
      return src[v];
    } else {
      return prob_from_logit(src[v], mx, p.inv_temp, z);
    }
  };
  if (!k_on && !p_on) {  // decided alike by every CTA of the cluster
    if constexpr (SRC == PSource::kProbs) {
      for (int v = s0 + threadIdx.x; v < s1; v += kSelThreads) p.p_out[row * V + v] = src[v];
    } else {
      if (rank == 0 && threadIdx.x == 0) p.sel[row] = SelRow{0u, V, 0ull};
    }
    return;
  }

  // probability keys of this CTA's slice, and the slice's mass
  unsigned long long local = 0;
  constexpr int kUnroll = 8;  // independent loads in flight per thread
  for (int i0 = threadIdx.x; i0 < n; i0 += kUnroll * kSelThreads) {
    float pv[kUnroll];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int i = i0 + j * kSelThreads;
      pv[j] = i < n ? base_prob(s0 + i) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int i = i0 + j * kSelThreads;
      if (i < n) {
        const uint32_t key = prob_key(pv[j]);
        keys[i] = key;
        local += key_mass(key);
      }
    }
  }
  local = block_sum_u64(local, sh);
  if (threadIdx.x == 0) {
    sh.total = local;
    sh.cut = V;
  }
  cluster.sync();
  if (threadIdx.x == 0) {
    unsigned long long S = 0;
    for (int r = 0; r < csize; ++r) S += cluster.map_shared_rank(&sh, r)->total;
    sh.all_total = S;
  }
  __syncthreads();

  int pass = 0;
  bool ok = sh.all_total > 0;
  SelectResult res{0u, 0ull, 0ull, 0u, true};
  unsigned long long keep = 0, Sk = sh.all_total;  // keep: how many of the keys == t are kept
  if (ok && k_on) {
    res = radix_select(cluster, sh, keys, n, false, (unsigned long long)K, pass);
    keep = (unsigned long long)K - res.above_c;
    Sk = res.above_m + keep * key_mass(res.t);
    ok = res.ok;
  }
  if (ok && p_on) {
    if (Sk == 0ull) {
      ok = false;
    } else {
      unsigned long long tau = (unsigned long long)ceil(__dmul_rn((double)TP, (double)Sk));
      if (tau < 1ull) tau = 1ull;
      res = radix_select(cluster, sh, keys, n, true, tau, pass);
      const unsigned long long Rt = key_mass(res.t);
      ok = res.ok && Rt > 0ull;
      if (ok) keep = (tau - res.above_m + Rt - 1ull) / Rt;  // >= 1: the mass above t is below tau
    }
  }
  const unsigned long long Z = ok ? res.above_m + keep * key_mass(res.t) : 0ull;

  // index cut among the keys equal to the threshold
  if (Z != 0ull && keep < res.tie_cnt) {
    unsigned long long mine = 0;
    for (int i = threadIdx.x; i < n; i += kSelThreads) mine += keys[i] == res.t;
    mine = block_sum_u64(mine, sh);
    if (threadIdx.x == 0) sh.ties = (unsigned int)mine;
    cluster.sync();
    if (threadIdx.x == 0) {
      unsigned int before = 0;
      for (int r = 0; r < rank; ++r) before += cluster.map_shared_rank(&sh, r)->ties;
      sh.ties_before = before;
    }
    __syncthreads();
    const long long need0 = (long long)keep - sh.ties_before;  // 1-based rank of the cut in this slice
    if (need0 >= 1 && need0 <= (long long)mine) {
      long long need = need0;
      const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
      for (int base = 0; base < n && need > 0; base += kSelThreads) {
        const int i = base + threadIdx.x;
        const bool f = i < n && keys[i] == res.t;
        const uint32_t bal = __ballot_sync(0xffffffffu, f);
        if (lane == 0) sh.wc[warp] = __popc(bal);
        __syncthreads();
        int pre = __popc(bal & ((1u << lane) - 1u)), tot = 0;
        for (int w = 0; w < kSelWarps; ++w) {
          if (w < warp) pre += sh.wc[w];
          tot += sh.wc[w];
        }
        if (f && pre + 1 == need) {
          for (int r = 0; r < csize; ++r) *cluster.map_shared_rank(&sh.cut, r) = s0 + i;
        }
        need -= tot;
        __syncthreads();
      }
    }
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
  const SelRow s{res.t, sh.cut, Z};
  if constexpr (SRC == PSource::kProbs) {
    const double inv = sel_inv_z(s);
    for (int i = threadIdx.x; i < n; i += kSelThreads)
      p.p_out[row * V + s0 + i] = Z ? adjusted_prob(__uint_as_float(keys[i]), s0 + i, s, inv) : src[s0 + i];
  } else {
    if (rank == 0 && threadIdx.x == 0) p.sel[row] = s;
  }
}

template <PSource SRC>
cudaError_t set_select_attrs(size_t smem) {
  static size_t set_to = 0;
  if (smem <= set_to) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(select_kernel<SRC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) set_to = smem;
  return e;
}

}  // namespace

int select_max_vocab() { return kSelCluster * kSelMaxSlice; }

cudaError_t launch_select(const SelectParams& p, PSource src, int n_rows_or_wmax, int B, cudaStream_t st) {
  const int slice = (p.V + kSelCluster - 1) / kSelCluster;
  if (slice > kSelMaxSlice) return cudaErrorInvalidValue;
  const size_t smem = (size_t)slice * 4;
  if (src == PSource::kProbs) {
    if (cudaError_t e = set_select_attrs<PSource::kProbs>(smem)) return e;
    return launch_k_cluster(select_kernel<PSource::kProbs>, dim3(kSelCluster, n_rows_or_wmax, 1), dim3(kSelThreads),
                            smem, st, dim3(kSelCluster, 1, 1), p);
  }
  if (cudaError_t e = set_select_attrs<PSource::kLogits>(smem)) return e;
  return launch_k_cluster(select_kernel<PSource::kLogits>, dim3(kSelCluster, n_rows_or_wmax, B), dim3(kSelThreads),
                          smem, st, dim3(kSelCluster, 1, 1), p);
}

}  // namespace spec
