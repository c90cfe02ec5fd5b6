// Acceptance of the verify round: logits -> (argmax | softmax statistics) ->
// accept / resample / bonus -> commit.
//
// Greedy ("Per-step cost versus accepted tokens", "What SGLang actually runs";
// Lecture 6 "Optimizing Autoregressive Decode" section 7.4): compare each draft
// with the target argmax at its position, accept the longest matching prefix,
// and commit the target argmax at the first mismatch (or after the last draft).
//
// Sampled (Lecture 6 section 6.2, Leviathan Algorithm 1): accept x_i while
// u_i * q_i(x_i) < p_i(x_i) (fp32 product, no fused multiply-add); after a
// rejection at position n+1 draw from norm(max(0, p_{n+1} - q_{n+1})); after
// full acceptance draw the bonus from p_{gamma+1}.  The one final draw is an
// integer inverse CDF: masses R_v = floor(r_v * 2^40) as 64-bit integers, their
// exact sum S, target t = floor(floor(u * 2^24) * S / 2^24), answer = smallest v
// whose running sum exceeds t.  Integer sums do not depend on the reduction
// order, so the draw is reproducible bit for bit against a sequential CPU
// computation on the same probabilities.  If the residual has no mass on that
// grid the draw falls back to p at the same row; a row of p without mass on the
// grid (not a distribution: only given probabilities can be one) gives token 0.
// The round kernel below takes these decisions for model rounds (from the LM
// head's tile statistics) and for given probabilities (standalone entry point).
//
// Tree (section 10.3): walk from the root to the child whose token equals the
// argmax at the current node (lowest node index on ties), then move the
// accepted path's KV into consecutive slots and cut the cache.
#include <cooperative_groups.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "kvstate.cuh"
#include "launch.cuh"
#include "sampling.cuh"

namespace cg = cooperative_groups;

namespace spec {

namespace {

constexpr int kAccThreads = 1024;

// Accept tests of drafts 1..gamma, evaluated side by side by one warp (lane i
// tests draft i: 1 accept, 0 reject, -1 invalid token) instead of one after the
// other: the accepted prefix ends at the first failing test, and an invalid token
// there is flagged (the tests past it cannot change the outcome).  All lanes of
// the calling warp return the prefix length; gamma < 32.
template <typename Test>
SPEC_DEVICE_INLINE int accepted_prefix(int gamma, int lane, int* status, Test&& test) {
  const bool mine = lane >= 1 && lane <= gamma;
  const int r = mine ? test(lane) : 1;
  const unsigned fail = __ballot_sync(0xffffffffu, mine && r != 1);
  if (fail == 0u) return gamma;
  const int f = __ffs(fail) - 1;  // first failing draft
  if (lane == f && r < 0) set_status(status, SPEC_ERR_INVALID_ARG);
  return f - 1;
}

struct ArgMax {
  float v;
  int i;
};

SPEC_DEVICE_INLINE ArgMax better(ArgMax a, ArgMax b) {
  if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
  return a;
}

SPEC_DEVICE_INLINE ArgMax warp_argmax(ArgMax a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ArgMax b;
    b.v = __shfl_xor_sync(0xffffffffu, a.v, o);
    b.i = __shfl_xor_sync(0xffffffffu, a.i, o);
    a = better(a, b);
  }
  return a;
}

// One block per row: argmax (lowest index on ties) and, for sampled rounds, the
// row max and sum_v exp((l_v - max) / T).
__global__ void __launch_bounds__(kAccThreads) row_stats_kernel(const float* rows, int V, float inv_temp, int sampled,
                                                                int32_t* argmax, float* row_max, float* row_sum) {
  __shared__ ArgMax sa[32];
  __shared__ float sf[32];
  pdl_wait();
  pdl_launch_dependents();
  const float* r = rows + (long long)blockIdx.x * V;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ArgMax best{-INFINITY, 0x7fffffff};
  for (int v = threadIdx.x; v < V; v += kAccThreads) best = better(best, ArgMax{r[v], v});
  best = warp_argmax(best);
  if (lane == 0) sa[warp] = best;
  __syncthreads();
  if (warp == 0) {
    ArgMax a = lane < kAccThreads / 32 ? sa[lane] : ArgMax{-INFINITY, 0x7fffffff};
    a = warp_argmax(a);
    if (lane == 0) sa[0] = a;
  }
  __syncthreads();
  best = sa[0];
  if (threadIdx.x == 0) argmax[blockIdx.x] = best.i == 0x7fffffff ? 0 : best.i;
  if (!sampled) return;
  const float mx = best.v;
  float s = 0.f;
  for (int v = threadIdx.x; v < V; v += kAccThreads) s += expf((r[v] - mx) * inv_temp);
  s = warp_sum(s);
  if (lane == 0) sf[warp] = s;
  __syncthreads();
  if (warp == 0) {
    float t = lane < kAccThreads / 32 ? sf[lane] : 0.f;
    t = warp_sum(t);
    if (lane == 0) {
      row_max[blockIdx.x] = mx;
      row_sum[blockIdx.x] = t;
    }
  }
}

// Exclusive block scan of 64-bit values; returns the prefix, total via *total.
SPEC_DEVICE_INLINE unsigned long long block_exscan_u64(unsigned long long v, unsigned long long* sh,
                                                       unsigned long long* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    unsigned long long w = lane < nw ? sh[lane] : 0ull;
    unsigned long long winc = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, winc, o);
      if (lane >= o) winc += y;
    }
    if (lane < nw) sh[lane] = winc - w;  // exclusive warp offsets
    if (lane == nw - 1) sh[32] = winc;
  }
  __syncthreads();
  const unsigned long long pre = sh[warp] + inc - v;
  *total = sh[32];
  __syncthreads();
  return pre;
}

// Standalone greedy acceptance: one block per sequence takes the argmax of its
// W rows (or reads them from row_argmax), then the longest matching prefix.
__global__ void __launch_bounds__(kAccThreads) accept_greedy_kernel(const __grid_constant__ AcceptParams p) {
  __shared__ int s_n, s_tok;
  __shared__ int s_am[kMaxWidth];
  __shared__ ArgMax s_red[32];
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int W = p.gamma + 1;
  const int V = p.V;
  const long long row0 = (long long)b * W;
  auto xdraft = [&](int i) -> int { return p.tok[(long long)b * p.gamma + i - 1]; };
  if (p.row_argmax == nullptr) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int row = 0; row < W; ++row) {
      const float* r = p.rows + (row0 + row) * V;
      ArgMax best{-INFINITY, 0x7fffffff};
      for (int v = threadIdx.x; v < V; v += kAccThreads) best = better(best, ArgMax{r[v], v});
      best = warp_argmax(best);
      if (lane == 0) s_red[warp] = best;
      __syncthreads();
      if (warp == 0) {
        ArgMax a = lane < kAccThreads / 32 ? s_red[lane] : ArgMax{-INFINITY, 0x7fffffff};
        a = warp_argmax(a);
        if (lane == 0) s_am[row] = a.i == 0x7fffffff ? 0 : a.i;
      }
      __syncthreads();
    }
  }
  auto am = [&](int row) -> int { return p.row_argmax ? p.row_argmax[row0 + row] : s_am[row]; };
  if (threadIdx.x < 32) {
    const int n = accepted_prefix(p.gamma, threadIdx.x, nullptr, [&](int i) -> int {
      const int x = xdraft(i);
      if (x < 0 || x >= V) return -1;
      return x == am(i - 1) ? 1 : 0;
    });
    if (threadIdx.x == 0) {
      s_n = n;
      s_tok = am(n);
    }
  }
  __syncthreads();
  const int n = s_n;
  const int tok_final = s_tok;
  for (int j = threadIdx.x; j < W; j += kAccThreads)
    p.committed[row0 + j] = j < n ? xdraft(j + 1) : (j == n ? tok_final : -1);
  if (threadIdx.x == 0) {
    p.accepted[b] = n;
    p.bonus[b] = tok_final;
  }
}

// Merge the LM head's per-128-column statistics of window row `row`: row max,
// lowest index attaining it, and Z = sum_v exp((l_v - max) / T).  One warp per row;
// lane l takes tiles l, l + 32, ... in ascending order, with eight tiles' loads in
// flight at a time (the loads do not depend on each other), then a fixed shuffle
// tree: the same order on every run, so Z is reproducible.
SPEC_DEVICE_INLINE void merge_row_stats(const RoundAcceptParams& p, long long m, bool sampled, float* out_max,
                                        float* out_z, int* out_arg) {
  constexpr int U = 8;
  const int lane = threadIdx.x & 31;
  float mx = -INFINITY;
  int am = 0x7fffffff;
  for (int t0 = lane; t0 < p.n_tiles; t0 += 32 * U) {
    float v[U];
    int a[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int t = t0 + 32 * k;
      v[k] = t < p.n_tiles ? p.tstat_max[(long long)t * p.tstat_stride + m] : -INFINITY;
      a[k] = t < p.n_tiles ? p.tstat_arg[(long long)t * p.tstat_stride + m] : 0x7fffffff;
    }
#pragma unroll
    for (int k = 0; k < U; ++k)
      if (v[k] > mx || (v[k] == mx && a[k] < am)) {
        mx = v[k];
        am = a[k];
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
  float z = 0.f;
  if (sampled) {
    for (int t0 = lane; t0 < p.n_tiles; t0 += 32 * U) {
      float tm[U], ts[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int t = t0 + 32 * k;
        tm[k] = t < p.n_tiles ? p.tstat_max[(long long)t * p.tstat_stride + m] : 0.f;
        ts[k] = t < p.n_tiles ? p.tstat_sum[(long long)t * p.tstat_stride + m] : 0.f;
      }
#pragma unroll
      for (int k = 0; k < U; ++k)
        if (t0 + 32 * k < p.n_tiles) z += ts[k] * expf((tm[k] - mx) * p.inv_temp);
    }
    z = warp_sum(z);
  }
  if (lane == 0) {
    *out_max = mx;
    *out_z = z;
    *out_arg = am == 0x7fffffff ? 0 : am;
  }
}

// One verify round's acceptance and commit for sequence blockIdx.y.  Sampled
// rounds run as a cluster of kDrawCluster CTAs that split the vocabulary for
// the final draw; greedy rounds use one CTA.
//
// SRC = kProbs: the same acceptance on given target probabilities (p.probs, rows
// of sequence b at b * (gamma + 1)) and drafts p.x, without a commit -- the
// standalone entry point, so that this kernel's decisions can be checked on
// identical inputs.
template <bool SAMPLED, PSource SRC = PSource::kLogits>
__global__ void __launch_bounds__(kAccThreads) accept_round_kernel(const __grid_constant__ RoundAcceptParams p) {
  __shared__ float s_max[kMaxWidth], s_z[kMaxWidth];
  __shared__ int s_am[kMaxWidth];
  __shared__ int s_n;
  __shared__ unsigned long long s_scan[33];
  __shared__ unsigned long long s_total;
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.y;
  const int V = p.V;
  const int Wmax = p.gamma + 1;                  // stride of u and committed
  const int Wfwd = p.seq_wlen ? p.seq_wlen[b] : Wmax;  // rows the forward scored for this sequence
  const int W = p.cap ? max(1, min(p.cap[b], Wfwd)) : Wfwd;  // rows the acceptance may use
  const int gamma = W - 1;
  const long long row0 = p.seq_rowoff ? p.seq_rowoff[b] : (long long)b * Wmax;
  const long long urow = (long long)b * Wmax;
  const int warp = threadIdx.x >> 5;

  if constexpr (SRC == PSource::kLogits) {
    if (warp < W) merge_row_stats(p, row0 + warp, SAMPLED, &s_max[warp], &s_z[warp], &s_am[warp]);
    __syncthreads();
  }
  // top-k / top-p: the selection kernel's statistics and kept set of each row
  __shared__ SelRow s_sel[kMaxWidth];
  __shared__ double s_inv[kMaxWidth];
  const bool adjust = SAMPLED && SRC == PSource::kLogits && p.sel != nullptr;
  if (adjust) {
    if (threadIdx.x < W) {
      const long long r = row0 + threadIdx.x;
      s_max[threadIdx.x] = p.sel_max[r];
      s_z[threadIdx.x] = p.sel_z[r];
      s_sel[threadIdx.x] = p.sel[r];
      s_inv[threadIdx.x] = sel_inv_z(s_sel[threadIdx.x]);
    }
    __syncthreads();
  }

  auto prob = [&](int row, int v) -> float {
    if constexpr (SRC == PSource::kProbs) {
      return p.probs[(row0 + row) * V + v];
    } else {
      const float pv = prob_from_logit(p.logits[(row0 + row) * V + v], s_max[row], p.inv_temp, s_z[row]);
      return adjust ? adjusted_prob(pv, v, s_sel[row], s_inv[row]) : pv;
    }
  };
  auto xdraft = [&](int i) -> int {  // x_i = window row i, or the given drafts
    return p.x ? p.x[(long long)b * p.gamma + i - 1] : p.tok[row0 + i];
  };

  if (warp == 0) {
    const int n = accepted_prefix(gamma, threadIdx.x, p.status, [&](int i) -> int {
      const int x = xdraft(i);
      if (x < 0 || x >= V) return -1;
      if constexpr (SAMPLED) {
        const float qx = p.q[((long long)b * p.gamma + (i - 1)) * V + x];
        return __fmul_rn(p.u[urow + i - 1], qx) < prob(i - 1, x) ? 1 : 0;
      } else {
        return x == s_am[i - 1] ? 1 : 0;
      }
    });
    if (threadIdx.x == 0) s_n = n;
  }
  __syncthreads();
  const int n = s_n;

  auto finish = [&](int tok_final) {  // one thread of the whole cluster
    for (int j = 0; j < Wmax; ++j) p.committed[urow + j] = j < n ? xdraft(j + 1) : (j == n ? tok_final : -1);
    p.accepted[b] = n;
    p.bonus[b] = tok_final;
    // a sequence whose window was refused (bad or repeated id, no pages) keeps
    // its length and pages
    if (p.seq_ids && (!p.seq_ok || p.seq_ok[b])) {
      const int s = p.seq_ids[b];
      if (s >= 0 && s < p.max_batch)
        truncate_seq(s, min(p.seq_len[s] + 1 + n, p.max_pages * kPage), p.seq_len, p.seq_npages, p.page_table,
                     p.max_pages, p.free_bits);
    }
  };

  if constexpr (!SAMPLED) {
    if (threadIdx.x == 0) finish(s_am[n]);
    return;
  } else {
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int csize = (int)cluster.num_blocks();
    const bool rejected = n < gamma;
    const float* qn = rejected ? p.q + ((long long)b * p.gamma + n) * V : nullptr;
    // this CTA's vocabulary slice, then this thread's sub-slice
    const int slice = (V + csize - 1) / csize;
    const int s0 = min(V, rank * slice), s1 = min(V, s0 + slice);
    const int chunk = (s1 - s0 + kAccThreads - 1) / kAccThreads;
    const int v0 = min(s1, s0 + (int)threadIdx.x * chunk), v1 = min(s1, v0 + chunk);
    const unsigned long long m = (unsigned long long)floorf(p.u[urow + gamma] * 16777216.0f);
    unsigned long long* tot_remote[kMaxDrawCluster];
    for (int pass = 0; pass < 2; ++pass) {
      const bool use_resid = rejected && pass == 0;
      auto mass = [&](int v) -> unsigned long long {
        const float pv = prob(n, v);
        const float r = use_resid ? fmaxf(0.f, pv - qn[v]) : pv;
        return (unsigned long long)floorf(r * 1099511627776.0f);  // r * 2^40, exact
      };
      unsigned long long local = 0;
      for (int v = v0; v < v1; ++v) local += mass(v);
      unsigned long long cta_total;
      const unsigned long long pre = block_exscan_u64(local, s_scan, &cta_total);
      if (threadIdx.x == 0) s_total = cta_total;
      cluster.sync();
      unsigned long long S = 0, before = 0;
      for (int r = 0; r < csize; ++r) {
        tot_remote[r] = cluster.map_shared_rank(&s_total, r);
        const unsigned long long tr = *tot_remote[r];
        if (r < rank) before += tr;
        S += tr;
      }
      cluster.sync();  // totals read before the next pass may overwrite them
      if (S == 0ull) {
        if (!use_resid) {  // p itself without mass on the grid: cannot happen for a distribution
          if (rank == 0 && threadIdx.x == 0) finish(0);
          break;
        }
        continue;  // residual without mass on the grid: draw from p at the same row
      }
      // t = floor(m * S / 2^24) with a 128-bit product (m < 2^24, S < 2^58)
      const unsigned long long hi = __umul64hi(m, S), lo = m * S;
      const unsigned long long t = (hi << 40) | (lo >> 24);
      const unsigned long long gpre = before + pre;
      if (local > 0 && gpre <= t && t < gpre + local) {
        unsigned long long run = gpre;
        for (int v = v0; v < v1; ++v) {
          run += mass(v);
          if (run > t) {
            finish(v);
            break;
          }
        }
      }
      break;
    }
  }
}

// Commit an accepted tree path of sequence b (the whole block calls it): move the
// path's KV (all layers, K and V) from slot L + node to slot L + depth, depth by
// depth, then cut the cache to L + 1 + n and record the round's outputs.  The
// destination L + d of depth d is never the source of a later depth (a node at
// depth d' has index >= d' > d), but it can be the source of an earlier one, so the
// depths run in order with a barrier between them.
SPEC_DEVICE_INLINE void commit_tree_path(const TreeParams& p, int b, const int* path, int n, int tok_final) {
  const int s = p.seq_ids[b];
  // a refused window (bad or repeated id, no pages; flagged by the prepare kernel)
  // moves no KV and keeps the sequence's length and pages
  const bool ok = s >= 0 && s < p.max_batch && (!p.seq_ok || p.seq_ok[b]);
  const int L = ok ? p.seq_len[s] : 0;
  const int vec_per_head = p.hd / 8;  // 16-byte vectors
  const int per_tok = p.n_layers * p.Hkv * vec_per_head;
  for (int d = 1; d <= n && ok; ++d) {
    const int src_t = L + path[d - 1], dst_t = L + d;
    if (src_t / kPage < p.max_pages) {
      const int src_pg = p.page_table[(long long)s * p.max_pages + src_t / kPage];
      const int dst_pg = p.page_table[(long long)s * p.max_pages + dst_t / kPage];
      if (src_pg >= 0 && dst_pg >= 0 && src_t != dst_t) {
        for (int r = threadIdx.x; r < per_tok; r += blockDim.x) {
          const int vec = r % vec_per_head;
          const int kvh = (r / vec_per_head) % p.Hkv;
          const int layer = r / (vec_per_head * p.Hkv);
          const long long src =
              ((((long long)layer * p.num_pages + src_pg) * p.Hkv + kvh) * kPage + src_t % kPage) * p.hd;
          const long long dst =
              ((((long long)layer * p.num_pages + dst_pg) * p.Hkv + kvh) * kPage + dst_t % kPage) * p.hd;
          reinterpret_cast<uint4*>(p.kpool + dst)[vec] = reinterpret_cast<const uint4*>(p.kpool + src)[vec];
          reinterpret_cast<uint4*>(p.vpool + dst)[vec] = reinterpret_cast<const uint4*>(p.vpool + src)[vec];
        }
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.accepted[b] = n;
    p.bonus[b] = tok_final;
    if (ok)
      truncate_seq(s, min(L + 1 + n, p.max_pages * kPage), p.seq_len, p.seq_npages, p.page_table, p.max_pages,
                   p.free_bits);
  }
}

__global__ void __launch_bounds__(kAccThreads) accept_tree_kernel(const __grid_constant__ TreeParams p) {
  __shared__ int s_path[kMaxWidth];
  __shared__ int s_n, s_tok;
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int N = p.N;
  const long long row0 = (long long)b * N;
  __shared__ float s_mx[kMaxWidth], s_z[kMaxWidth];
  __shared__ int s_am[kMaxWidth];
  {
    const int warp = threadIdx.x >> 5;
    if (warp < N) merge_row_stats(p.stats, row0 + warp, false, &s_mx[warp], &s_z[warp], &s_am[warp]);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int v = 0, k = 0, a = 0;
    while (true) {
      a = s_am[v];
      int nxt = -1;
      for (int c = 1; c < N; ++c) {
        if (p.parent[c] == v && p.tok[row0 + c] == a) {
          nxt = c;
          break;
        }
      }
      if (nxt < 0) break;
      s_path[k++] = nxt;
      v = nxt;
    }
    s_n = k;
    s_tok = a;
  }
  __syncthreads();
  const int n = s_n;
  for (int j = threadIdx.x; j < N; j += kAccThreads)
    p.committed[row0 + j] = j < n ? p.tok[row0 + s_path[j]] : (j == n ? s_tok : -1);
  commit_tree_path(p, b, s_path, n, s_tok);
}

// Sum of a 64-bit per-thread value over the cluster: returns the total and, via
// *before, the sum of the CTAs of lower rank plus this thread's exclusive prefix in
// its CTA (thread order = vocabulary order).  Two cluster barriers.
SPEC_DEVICE_INLINE unsigned long long cluster_scan_u64(cg::cluster_group& cluster, unsigned long long local,
                                                       unsigned long long* s_scan, unsigned long long* s_total,
                                                       unsigned long long* before) {
  unsigned long long cta_total;
  const unsigned long long pre = block_exscan_u64(local, s_scan, &cta_total);
  if (threadIdx.x == 0) *s_total = cta_total;
  cluster.sync();
  const int rank = (int)cluster.block_rank();
  unsigned long long S = 0, lower = 0;
  for (int r = 0; r < (int)cluster.num_blocks(); ++r) {
    const unsigned long long tr = *cluster.map_shared_rank(s_total, r);
    if (r < rank) lower += tr;
    S += tr;
  }
  cluster.sync();  // totals read before the next use may overwrite them
  *before = lower + pre;
  return S;
}

// Sampled verification of a token tree (SpecInfer's multi-step speculative
// sampling = recursive rejection over the children of a node; Lecture 6
// "Optimizing Autoregressive Decode" section 10.3).  From the root, the children of
// the current node v are tried in node order: child c (token x) is accepted when
// fl32(u[c] q_v(x)) < p_cur(x), where p_cur starts as the target at v and after
// each rejection becomes the normalised residual max(0, p_cur - q) (masses
// R = floor(r 2^40), p = fl32(fl64(R) * fl64(1/Z)), Z the exact sum); q_v is the
// distribution the children were drawn from, or the one-hot of the child's own
// token for deterministic candidates.  After the last child of v is rejected the
// final token is drawn from that residual (integer inverse CDF with u[0]); at a
// node without children it is the bonus draw from the target at v.  One cluster of
// kDrawCluster CTAs per sequence splits the vocabulary for the residual sums and
// the draw; every CTA takes the same decisions from the same values.
template <PSource SRC>
__global__ void __launch_bounds__(kAccThreads) accept_tree_sampled_kernel(const __grid_constant__ TreeParams p) {
  __shared__ float s_max[kMaxWidth], s_z[kMaxWidth];
  __shared__ int s_am[kMaxWidth];
  __shared__ SelRow s_sel[kMaxWidth];
  __shared__ double s_sinv[kMaxWidth];
  __shared__ double s_rinv[kMaxWidth];  // 1/Z of each rejection at the current node (0: no mass, keep p)
  __shared__ int s_rtok[kMaxWidth];     // deterministic candidates: the rejected tokens
  __shared__ int s_path[kMaxWidth];
  __shared__ int s_flag;
  __shared__ unsigned long long s_scan[33], s_total;
  pdl_wait();
  pdl_launch_dependents();
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int csize = (int)cluster.num_blocks();
  const int b = blockIdx.y;
  const int N = p.N, V = p.V;
  const long long row0 = (long long)b * N;
  const RoundAcceptParams& st = p.stats;
  bool adjust = false;
  if constexpr (SRC == PSource::kLogits) {
    const int warp = threadIdx.x >> 5;
    if (warp < N) merge_row_stats(st, row0 + warp, true, &s_max[warp], &s_z[warp], &s_am[warp]);
    __syncthreads();
    adjust = st.sel != nullptr;
    if (adjust) {
      if (threadIdx.x < N) {
        const long long r = row0 + threadIdx.x;
        s_max[threadIdx.x] = st.sel_max[r];
        s_z[threadIdx.x] = st.sel_z[r];
        s_sel[threadIdx.x] = st.sel[r];
        s_sinv[threadIdx.x] = sel_inv_z(s_sel[threadIdx.x]);
      }
      __syncthreads();
    }
  }
  auto base_prob = [&](int node, int w) -> float {
    if constexpr (SRC == PSource::kProbs) {
      return p.probs[(row0 + node) * V + w];
    } else {
      const float pv = prob_from_logit(st.logits[(row0 + node) * V + w], s_max[node], st.inv_temp, s_z[node]);
      return adjust ? adjusted_prob(pv, w, s_sel[node], s_sinv[node]) : pv;
    }
  };
  auto q_at = [&](int v, int j, int w) -> float {
    return p.q ? p.q[(row0 + v) * V + w] : (w == s_rtok[j] ? 1.f : 0.f);
  };
  // the target at node v after r rejections, at token w
  auto cur_prob = [&](int v, int r, int w) -> float {
    float x = base_prob(v, w);
    for (int j = 0; j < r; ++j) {
      if (s_rinv[j] == 0.0) continue;
      const float rr = fmaxf(0.f, __fsub_rn(x, q_at(v, j, w)));
      x = __double2float_rn(__dmul_rn((double)grid_mass(rr), s_rinv[j]));
    }
    return x;
  };
  // this thread's contiguous vocabulary range
  const int slice = (V + csize - 1) / csize;
  const int s0 = min(V, rank * slice), s1 = min(V, s0 + slice);
  const int chunk = (s1 - s0 + kAccThreads - 1) / kAccThreads;
  const int v0 = min(s1, s0 + (int)threadIdx.x * chunk), v1 = min(s1, v0 + chunk);
  const unsigned long long um = (unsigned long long)floorf(p.u[row0] * 16777216.0f);

  int v = 0, k = 0;
  while (true) {
    int r = 0, moved = -1;
    bool last_rejected = false;
    int n_children = 0;
    for (int c = 1; c < N; ++c) n_children += p.parent[c] == v;
    int seen = 0;
    for (int c = 1; c < N; ++c) {
      if (p.parent[c] != v) continue;
      ++seen;
      const int x = p.tok[row0 + c];
      if (threadIdx.x == 0) {
        bool acc = false;
        if (x < 0 || x >= V) {
          if (rank == 0) set_status(st.status, SPEC_ERR_INVALID_ARG);
        } else {
          const float qx = p.q ? p.q[(row0 + v) * V + x] : 1.f;
          acc = __fmul_rn(p.u[row0 + c], qx) < cur_prob(v, r, x);
        }
        s_flag = acc;
        if (!acc && !p.q) s_rtok[r] = x;
      }
      __syncthreads();
      if (s_flag) {
        moved = c;
        break;
      }
      if (seen == n_children) {
        last_rejected = true;
        break;
      }
      // normaliser of the residual after this rejection
      unsigned long long local = 0;
      for (int w = v0; w < v1; ++w) local += grid_mass(fmaxf(0.f, __fsub_rn(cur_prob(v, r, w), q_at(v, r, w))));
      unsigned long long before;
      const unsigned long long Z = cluster_scan_u64(cluster, local, s_scan, &s_total, &before);
      if (threadIdx.x == 0) s_rinv[r] = Z ? __ddiv_rn(1.0, (double)Z) : 0.0;
      __syncthreads();
      ++r;
    }
    if (moved >= 0) {
      if (threadIdx.x == 0) s_path[k] = moved;
      __syncthreads();
      ++k;
      v = moved;
      continue;
    }
    // final draw: the residual after the last rejection, or the target at a node
    // without children; without mass on the grid, the current target
    bool drawn = false;  // decided alike by every CTA (the totals are cluster-wide)
    for (int pass = 0; pass < 2 && !drawn; ++pass) {
      const bool resid = last_rejected && pass == 0;
      if (pass == 1 && !last_rejected) break;
      auto mass = [&](int w) -> unsigned long long {
        const float pc = cur_prob(v, r, w);
        return grid_mass(resid ? fmaxf(0.f, __fsub_rn(pc, q_at(v, r, w))) : pc);
      };
      unsigned long long local = 0;
      for (int w = v0; w < v1; ++w) local += mass(w);
      unsigned long long before;
      const unsigned long long S = cluster_scan_u64(cluster, local, s_scan, &s_total, &before);
      if (S == 0ull) continue;
      // t = floor(m * S / 2^24) with a 128-bit product (m < 2^24, S < 2^58)
      const unsigned long long hi = __umul64hi(um, S), lo = um * S;
      const unsigned long long t = (hi << 40) | (lo >> 24);
      drawn = true;  // the token is found by the thread whose range holds t
      if (local > 0 && before <= t && t < before + local) {
        unsigned long long run = before;
        for (int w = v0; w < v1; ++w) {
          run += mass(w);
          if (run > t) {
            s_flag = w;
            break;
          }
        }
        // this thread writes the round's outputs
        for (int j = 0; j < N; ++j)
          p.committed[row0 + j] = j < k ? p.tok[row0 + s_path[j]] : (j == k ? s_flag : -1);
        if (p.path)
          for (int j = 0; j < N; ++j) p.path[row0 + j] = j < k ? s_path[j] : -1;
        p.accepted[b] = k;
        p.bonus[b] = s_flag;
      }
    }
    if (!drawn && rank == 0 && threadIdx.x == 0) {  // no mass anywhere: token 0
      for (int j = 0; j < N; ++j) p.committed[row0 + j] = j < k ? p.tok[row0 + s_path[j]] : (j == k ? 0 : -1);
      if (p.path)
        for (int j = 0; j < N; ++j) p.path[row0 + j] = j < k ? s_path[j] : -1;
      p.accepted[b] = k;
      p.bonus[b] = 0;
    }
    break;
  }
}

// KV commit of the sampled tree round (one block per sequence).
__global__ void __launch_bounds__(kAccThreads) tree_commit_kernel(const __grid_constant__ TreeParams p) {
  __shared__ int s_path[kMaxWidth];
  __shared__ int s_n, s_tok;
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  if (threadIdx.x < p.N) s_path[threadIdx.x] = p.path[(long long)b * p.N + threadIdx.x];
  if (threadIdx.x == 0) {
    s_n = p.accepted[b];
    s_tok = p.bonus[b];
  }
  __syncthreads();
  commit_tree_path(p, b, s_path, s_n, s_tok);
}

}  // namespace

cudaError_t launch_row_stats(const float* rows, int n_rows, int V, float inv_temp, bool sampled, int32_t* argmax,
                             float* row_max, float* row_sum, cudaStream_t st) {
  return launch_k(row_stats_kernel, dim3(n_rows), dim3(kAccThreads), 0, st, rows, V, inv_temp, sampled ? 1 : 0,
                  argmax, row_max, row_sum);
}

cudaError_t launch_accept_greedy(const AcceptParams& p, cudaStream_t st) {
  return launch_k(accept_greedy_kernel, dim3(p.B), dim3(kAccThreads), 0, st, p);
}

cudaError_t launch_accept_round(const RoundAcceptParams& p, bool sampled, cudaStream_t st) {
  if (!sampled) return launch_k(accept_round_kernel<false>, dim3(1, p.B), dim3(kAccThreads), 0, st, p);
  return launch_k_cluster(accept_round_kernel<true>, dim3(kDrawCluster, p.B), dim3(kAccThreads), 0, st,
                          dim3(kDrawCluster, 1, 1), p);
}

cudaError_t launch_accept_round_probs(const RoundAcceptParams& p, cudaStream_t st) {
  // one cluster per sequence along grid y (at most 65535): larger batches in chunks
  constexpr int kChunk = 65535;
  const int W = p.gamma + 1;
  for (int b0 = 0; b0 < p.B; b0 += kChunk) {
    RoundAcceptParams c = p;
    c.B = std::min(kChunk, p.B - b0);
    c.probs = p.probs + (long long)b0 * W * p.V;
    if (p.q) c.q = p.q + (long long)b0 * p.gamma * p.V;
    if (p.x) c.x = p.x + (long long)b0 * p.gamma;
    c.u = p.u + (long long)b0 * W;
    c.accepted = p.accepted + b0;
    c.committed = p.committed + (long long)b0 * W;
    c.bonus = p.bonus + b0;
    cudaError_t e = launch_k_cluster(accept_round_kernel<true, PSource::kProbs>, dim3(kDrawCluster, c.B),
                                     dim3(kAccThreads), 0, st, dim3(kDrawCluster, 1, 1), c);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_accept_tree_sampled(const TreeParams& p, cudaStream_t st) {
  cudaError_t e;
  if (p.probs)
    e = launch_k_cluster(accept_tree_sampled_kernel<PSource::kProbs>, dim3(kDrawCluster, p.B), dim3(kAccThreads), 0,
                         st, dim3(kDrawCluster, 1, 1), p);
  else
    e = launch_k_cluster(accept_tree_sampled_kernel<PSource::kLogits>, dim3(kDrawCluster, p.B), dim3(kAccThreads),
                         0, st, dim3(kDrawCluster, 1, 1), p);
  if (e != cudaSuccess || !p.path || !p.seq_ids) return e;
  return launch_k(tree_commit_kernel, dim3(p.B), dim3(kAccThreads), 0, st, p);
}

cudaError_t launch_accept_tree(const TreeParams& p, cudaStream_t st) {
  return launch_k(accept_tree_kernel, dim3(p.B), dim3(kAccThreads), 0, st, p);
}

// ------------------------------------------------- allocation-free greedy accept
// Scratch of spec_accept_greedy_noalloc: the argmax of every logits row, written
// by the row-statistics kernel and read by the acceptance kernel.  It lives in
// this library's own device memory (every GPU that loads the library holds it
// until the process exits), so the entry point never allocates.
constexpr int kNoAllocMaxRows = 4096;
static __device__ __align__(256) int32_t g_noalloc_argmax[kNoAllocMaxRows];

namespace {

// Device address of the scratch array on the current device.  Host code cannot
// use the array's name as a device pointer, so the address is looked up once per
// device (with that device current) and cached.
cudaError_t noalloc_scratch(int32_t** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static int32_t* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_argmax);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<int32_t*>(p);
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace

}  // namespace spec

extern "C" spec_status spec_accept_greedy_noalloc(int32_t B, int32_t gamma, int32_t V, const float* logits,
                                                  const int32_t* x, int32_t* accepted, int32_t* committed,
                                                  int32_t* bonus, void* stream) {
  using namespace spec;
  if (B < 1 || gamma < 0 || gamma + 1 > kMaxWidth || V < 1) {
    record_error("spec_accept_greedy_noalloc: bad shape");
    return SPEC_ERR_INVALID_ARG;
  }
  if ((long long)B * (gamma + 1) > kNoAllocMaxRows) {
    record_error("spec_accept_greedy_noalloc: B*(gamma+1) exceeds the fixed scratch of 4096 rows");
    return SPEC_ERR_INVALID_ARG;
  }
  if (!logits || (gamma > 0 && !x) || !accepted || !committed || !bonus) {
    record_error("spec_accept_greedy_noalloc: NULL argument");
    return SPEC_ERR_INVALID_ARG;
  }
  int32_t* scratch = nullptr;
  cudaError_t e = noalloc_scratch(&scratch);
  if (e != cudaSuccess) {
    record_error(cudaGetErrorString(e));
    return SPEC_ERR_CUDA;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // every row's argmax is rewritten before it is read, so nothing needs clearing
  e = launch_row_stats(logits, B * (gamma + 1), V, 1.f, false, scratch, nullptr, nullptr, st);
  if (e == cudaSuccess) {
    AcceptParams ap{};
    ap.B = B;
    ap.gamma = gamma;
    ap.V = V;
    ap.rows = logits;
    ap.tok = x;
    ap.row_argmax = scratch;
    ap.accepted = accepted;
    ap.committed = committed;
    ap.bonus = bonus;
    e = launch_accept_greedy(ap, st);
  }
  if (e != cudaSuccess) {
    record_error(cudaGetErrorString(e));
    return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}
