// Sequence-state kernels: round preparation (page allocation + row metadata),
// reset, the prefill commit, and the random KV fill used for long-context timing.
#include <algorithm>

#include "kvstate.cuh"
#include "launch.cuh"

namespace spec {

namespace {

// One warp.  Sequence b owns flat rows rowoff_b .. rowoff_b + W_b - 1; for its
// window row j: position L + depth[j] (RoPE), KV slot L + j.  Lengths, offsets,
// positions, the slots of windows whose pages already exist and the token checks
// are computed 32 sequences at a time; only the sequences that need new pages are
// then served one at a time, in batch order b = 0..B-1 (deterministic page
// assignment: the lowest free page first, as if every sequence were served in
// turn -- the others take no page).
//
// A batch that names a sequence id out of range, or the same id twice, is refused
// as a whole (SPEC_ERR_INVALID_ARG): no page is taken, no KV slot is given out and
// every seq_ok[b] is 0, so the commit leaves every sequence as it was (two windows
// of one sequence would write the same slots and race on its length and pages).
// A sequence whose window cannot get its pages (SPEC_ERR_CAPACITY) gives back the
// pages this call took for it and gets seq_ok[b] = 0.  The status word keeps the
// first error in batch order (per sequence: a refused window length, then a
// capacity failure, then a token id out of range).
constexpr int kMaxBatch = 4096;  // max_batch <= 4096 (checked by the launcher)
constexpr int kMaxBatchWords = kMaxBatch / 32;
constexpr int kRankMax = 256;    // sequences ranked by cached length (more: batch order)
constexpr uint8_t kErrRefused = 1, kErrCapacity = 2, kErrToken = 4;
__global__ void __launch_bounds__(32) prepare_kernel(const __grid_constant__ PrepareParams p) {
  __shared__ uint32_t s_seen[kMaxBatchWords];
  __shared__ uint32_t s_alloc[kMaxBatchWords];  // bit b: sequence b needs pages this call
  __shared__ uint8_t s_err[kMaxBatch];          // kErr* bits of sequence b
  __shared__ int s_len[kRankMax];
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x;
  for (int i = lane; i < kMaxBatchWords; i += 32) {
    s_seen[i] = 0u;
    s_alloc[i] = 0u;
  }
  __syncwarp();
  bool bad_ids = false;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    bool bad = false;
    if (b < p.B) {
      const int s = p.seq_ids[b];
      if (s < 0 || s >= p.max_batch) {
        bad = true;
      } else {
        const uint32_t bit = 1u << (s & 31);
        bad = (atomicOr(&s_seen[s >> 5], bit) & bit) != 0u;  // seen before: a repeat
      }
    }
    bad_ids |= __any_sync(0xffffffffu, bad);
  }
  if (bad_ids && lane == 0) set_status(p.status, SPEC_ERR_INVALID_ARG);

  // Sequences b0 .. b0+31, one per lane.  Window lengths are clamped to [0, W] and
  // to the rows left (a length outside 1..W, or past total_rows, is refused), so the
  // row offset of b is min(total_rows, sum of the clamped lengths before it): an
  // exclusive prefix sum over the warp, carried from group to group.
  int rows_before = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    const bool in = b < p.B;
    const int s = in ? p.seq_ids[b] : -1;
    const int w_req = in ? (p.wlen ? p.wlen[b] : p.W) : 0;
    const int c = max(0, min(w_req, p.W));
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const int off = min(p.total_rows, rows_before + incl - c);
    rows_before = min(p.total_rows, rows_before + __shfl_sync(0xffffffffu, incl, 31));
    const int Wb = max(0, min(c, p.total_rows - off));
    uint8_t err = 0;
    if (in && (w_req < 1 || w_req > p.W || off + w_req > p.total_rows)) err |= kErrRefused;
    const bool sid_ok = in && s >= 0 && s < p.max_batch;
    const int L = sid_ok ? p.seq_len[s] : 0;
    bool ok = sid_ok && !bad_ids;
    bool alloc = false;
    if (ok) {
      const int need = (L + Wb + kPage - 1) / kPage;
      if (L + Wb > p.max_seq_len || need > p.max_pages) {
        ok = false;
        err |= kErrCapacity;
      } else {
        alloc = need > p.seq_npages[s];  // pages are taken below, in batch order
      }
    }
    if (in) {
      p.seq_start[b] = L;
      p.seq_wlen[b] = Wb;
      p.seq_rowoff[b] = off;
      p.seq_ok[b] = ok ? 1 : 0;
      for (int j = 0; j < Wb; ++j) {
        const int m = off + j;
        p.row_pos[m] = min(L + p.depth[j], p.max_seq_len - 1);
        int slot = -1;
        if (ok && !alloc) {
          const int t = L + j;
          slot = p.page_table[(long long)s * p.max_pages + t / kPage] * kPage + t % kPage;
        }
        p.row_slot[m] = slot;
        const int tk = p.tok[m];
        if (tk < 0 || tk >= p.vocab) err |= kErrToken;
      }
      s_err[b] = err;
    }
    const unsigned alloc_bits = __ballot_sync(0xffffffffu, alloc);
    if (lane == 0) s_alloc[b0 >> 5] = alloc_bits;
  }
  __syncwarp();

  // The sequences that need pages, in batch order (the whole warp serves each).
  const int n_words = (p.B + 31) >> 5;
  for (int w = 0; w < n_words; ++w) {
    uint32_t bits = s_alloc[w];
    while (bits) {
      const int b = (w << 5) + __ffs(bits) - 1;
      bits &= bits - 1u;
      const int s = p.seq_ids[b];
      const int L = p.seq_start[b], Wb = p.seq_wlen[b], off = p.seq_rowoff[b];
      const int npg0 = p.seq_npages[s];
      const bool ok = warp_ensure_pages(s, L + Wb, p.seq_npages, p.page_table, p.max_pages, p.free_bits, p.num_pages);
      if (lane == 0) {
        if (!ok) {
          release_pages_from(s, npg0, p.seq_npages, p.page_table, p.max_pages, p.free_bits);
          s_err[b] |= kErrCapacity;
        }
        p.seq_ok[b] = ok ? 1 : 0;
      }
      if (ok) {
        for (int j = lane; j < Wb; j += 32) {
          const int t = L + j;
          p.row_slot[off + j] = p.page_table[(long long)s * p.max_pages + t / kPage] * kPage + t % kPage;
        }
      }
      __syncwarp();
    }
  }

  // The first error in batch order.
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    const int e = b < p.B ? s_err[b] : 0;
    const int code = (e & kErrRefused)    ? SPEC_ERR_INVALID_ARG
                     : (e & kErrCapacity) ? SPEC_ERR_CAPACITY
                     : (e & kErrToken)    ? SPEC_ERR_INVALID_ARG
                                          : 0;
    const unsigned any = __ballot_sync(0xffffffffu, code != 0);
    if (any) {
      if (lane == __ffs(any) - 1) set_status(p.status, code);
      break;
    }
  }
  if (lane == 0 && rows_before != p.total_rows) set_status(p.status, SPEC_ERR_INVALID_ARG);

  // The attention's CTA groups go longest cache first: with more groups than one
  // wave, the short ones fill in behind the long ones instead of a long one
  // starting last.  Rank of b: the sequences with a longer cache, or an equal one
  // and a lower index (a permutation).  Up to kRankMax sequences; beyond, batch order.
  const bool rank = p.B <= kRankMax;
  if (rank)
    for (int b = lane; b < p.B; b += 32) s_len[b] = p.seq_start[b];
  __syncwarp();
  for (int b = lane; b < p.B; b += 32) {
    int r = b;
    if (rank) {
      const int Lb = s_len[b];
      r = 0;
      for (int j = 0; j < p.B; ++j) {
        const int Lj = s_len[j];
        r += (Lj > Lb || (Lj == Lb && j < b)) ? 1 : 0;
      }
    }
    p.seq_order[r] = b;
  }
}

__global__ void seq_reset_kernel(const int32_t* seq_ids, int n, int32_t* seq_len, int32_t* seq_npages,
                                 int32_t* page_table, uint32_t* free_bits, int max_pages) {
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x != 0) return;
  for (int i = 0; i < n; ++i) truncate_seq(seq_ids[i], 0, seq_len, seq_npages, page_table, max_pages, free_bits);
}

// Prefill windows commit every row: L <- L + W (refused windows: unchanged).
__global__ void commit_all_kernel(const int32_t* seq_ids, const int32_t* seq_ok, int B, int W, int max_batch,
                                  int32_t* seq_len) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int s = seq_ids[b];
  if (s >= 0 && s < max_batch && seq_ok[b]) seq_len[s] += W;
}

// Pages for each listed sequence, in list order (lowest free page first).
// relative == 0: the sequence gets exactly lens[i] cached tokens (length set).
// relative == 1: pages are reserved for lens[i] more tokens after the current
//                length (a prefill reserves its whole prompt up front, so page
//                assignment follows the caller's sequence order, not the order
//                in which prefill windows happen to run).  Length unchanged.
__global__ void __launch_bounds__(32) alloc_to_len_kernel(const int32_t* seq_ids, const int32_t* lens, int n,
                                                          int relative, int32_t* seq_len, int32_t* seq_npages,
                                                          int32_t* page_table, uint32_t* free_bits, int max_pages,
                                                          int num_pages, int max_batch, int* status) {
  pdl_wait();
  pdl_launch_dependents();
  for (int i = 0; i < n; ++i) {
    const int s = seq_ids[i];
    if (s < 0 || s >= max_batch) {
      if (threadIdx.x == 0) set_status(status, SPEC_ERR_INVALID_ARG);
      continue;
    }
    const int upto = relative ? seq_len[s] + lens[i] : lens[i];
    const int npg0 = seq_npages[s];
    const bool ok = warp_ensure_pages(s, upto, seq_npages, page_table, max_pages, free_bits, num_pages);
    if (threadIdx.x == 0) {
      if (!ok) {  // give back what this call took: the sequence keeps the pages it had
        set_status(status, SPEC_ERR_CAPACITY);
        release_pages_from(s, npg0, seq_npages, page_table, max_pages, free_bits);
      }
      if (!relative) seq_len[s] = ok ? lens[i] : 0;
    }
    __syncwarp();
  }
}

SPEC_DEVICE_INLINE uint64_t splitmix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

// Fill K and V of every allocated page of the listed sequences, all layers.
// grid: (pages, n_layers, n); each block writes one (layer, page) of one sequence.
__global__ void kv_fill_kernel(act_t* kpool, act_t* vpool, const int32_t* page_table,
                               const int32_t* seq_npages, int max_pages, const int32_t* seq_ids, int num_pages,
                               int Hkv, int hd, uint64_t seed, float scale) {
  pdl_wait();
  pdl_launch_dependents();
  const int s = seq_ids[blockIdx.z];
  const int layer = blockIdx.y;
  const int pi = blockIdx.x;
  if (pi >= seq_npages[s]) return;
  const int pg = page_table[(long long)s * max_pages + pi];
  if (pg < 0) return;
  const long long per_page = (long long)Hkv * kPage * hd;
  const long long base = ((long long)layer * num_pages + pg) * per_page;
  for (long long e = threadIdx.x; e < per_page; e += blockDim.x) {
    const uint64_t h = splitmix64(seed ^ (uint64_t)(base + e) * 0x2545F4914F6CDD1Dull);
    const float a = ((float)(uint32_t)(h & 0xffffffu) * (1.0f / 16777216.0f) * 2.f - 1.f) * scale;
    const float c = ((float)(uint32_t)((h >> 32) & 0xffffffu) * (1.0f / 16777216.0f) * 2.f - 1.f) * scale;
    kpool[base + e] = to_act(a);
    vpool[base + e] = to_act(c);
  }
}

// Copy caller-supplied K/V of sequence seq_id (tokens 0..n-1, [n_layers][n][Hkv][hd]
// fp16 each) into its pages.  grid: (pages of the sequence, n_layers); one block
// per (page, layer), 16-byte vectors.
__global__ void kv_write_kernel(act_t* kpool, act_t* vpool, const int32_t* page_table, int max_pages, int seq_id,
                                int n, const act_t* k, const act_t* v, int num_pages, int Hkv, int hd) {
  pdl_wait();
  pdl_launch_dependents();
  const int pi = blockIdx.x, layer = blockIdx.y;
  const int pg = page_table[(long long)seq_id * max_pages + pi];
  if (pg < 0) return;
  const int vec = hd / 8;
  const int t0 = pi * kPage;
  const int nt = min(kPage, n - t0);
  for (int e = threadIdx.x; e < nt * Hkv * vec; e += blockDim.x) {
    const int d8 = e % vec, h = (e / vec) % Hkv, t = e / (vec * Hkv);
    const long long src = (((long long)layer * n + t0 + t) * Hkv + h) * hd;
    const long long dst = ((((long long)layer * num_pages + pg) * Hkv + h) * kPage + t) * hd;
    reinterpret_cast<uint4*>(kpool + dst)[d8] = reinterpret_cast<const uint4*>(k + src)[d8];
    reinterpret_cast<uint4*>(vpool + dst)[d8] = reinterpret_cast<const uint4*>(v + src)[d8];
  }
}

__global__ void gather_tokens_kernel(const int32_t* tokens, int stride, const int32_t* perm, int k, int col0, int W,
                                     int32_t* out, const int32_t* seq_ids, int32_t* ids_out) {
  pdl_wait();
  pdl_launch_dependents();
  const int i = blockIdx.x;
  const int b = perm[i];
  for (int j = threadIdx.x; j < W; j += blockDim.x) out[i * W + j] = tokens[(long long)b * stride + col0 + j];
  if (threadIdx.x == 0) ids_out[i] = seq_ids[b];
}

__global__ void init_state_kernel(int32_t* seq_len, int32_t* seq_npages, int32_t* page_table, uint32_t* free_bits,
                                  int max_batch, int max_pages, int num_pages) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < max_batch) {
    seq_len[i] = 0;
    seq_npages[i] = 0;
  }
  if (i < (long long)max_batch * max_pages) page_table[i] = -1;
  const int nwords = (num_pages + 31) / 32;
  if (i < nwords) {
    const int lo = (int)i * 32;
    const int valid = min(32, num_pages - lo);
    free_bits[i] = valid >= 32 ? 0xffffffffu : ((1u << valid) - 1u);
  }
}

}  // namespace

cudaError_t launch_gather_tokens(const int32_t* tokens, int stride, const int32_t* perm, int k, int col0, int W,
                                 int32_t* out, const int32_t* seq_ids, int32_t* ids_out, cudaStream_t st) {
  return launch_k(gather_tokens_kernel, dim3(k), dim3(32), 0, st, tokens, stride, perm, k, col0, W, out, seq_ids,
                  ids_out);
}

cudaError_t launch_kv_write(act_t* kpool, act_t* vpool, const int32_t* page_table, int max_pages, int seq_id, int n,
                            const act_t* k, const act_t* v, int n_layers, int num_pages, int Hkv, int hd,
                            cudaStream_t st) {
  const int pages = (n + kPage - 1) / kPage;
  if (pages == 0) return cudaSuccess;
  return launch_k(kv_write_kernel, dim3(pages, n_layers), dim3(256), 0, st, kpool, vpool, page_table, max_pages,
                  seq_id, n, k, v, num_pages, Hkv, hd);
}

cudaError_t launch_init_state(int32_t* seq_len, int32_t* seq_npages, int32_t* page_table, uint32_t* free_bits,
                              int max_batch, int max_pages, int num_pages, cudaStream_t st) {
  const long long n = std::max<long long>({(long long)max_batch * max_pages, (long long)max_batch,
                                           (long long)(num_pages + 31) / 32});
  init_state_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(seq_len, seq_npages, page_table, free_bits,
                                                                  max_batch, max_pages, num_pages);
  return cudaGetLastError();
}

cudaError_t launch_prepare(const PrepareParams& p, cudaStream_t st) {
  if (p.B < 1 || p.B > kMaxBatch || p.W < 1 || p.W > 16) return cudaErrorInvalidValue;
  return launch_k(prepare_kernel, dim3(1), dim3(32), 0, st, p);
}

// A bounded wait that nothing completes: phase 0 of a fresh mbarrier needs one
// arrival and none comes, so the wait runs out after `budget` SM cycles and
// records SPEC_ERR_TIMEOUT -- the path every pipeline wait of the library takes
// when its partner stalls, taken here on purpose and with nothing else in flight.
__global__ void wait_probe_kernel(int* status, unsigned long long budget) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, status, budget);
}

cudaError_t launch_wait_probe(int* status, unsigned long long budget, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(status, budget);
  return cudaGetLastError();
}

cudaError_t launch_seq_reset(const ResetParams& p, cudaStream_t st) {
  return launch_k(seq_reset_kernel, dim3(1), dim3(32), 0, st, p.seq_ids, p.n, p.seq_len, p.seq_npages, p.page_table,
                  p.free_bits, p.max_pages);
}

cudaError_t launch_commit_all(const int32_t* seq_ids, const int32_t* seq_ok, int B, int W, int max_batch,
                              int32_t* seq_len, cudaStream_t st) {
  return launch_k(commit_all_kernel, dim3((B + 127) / 128), dim3(128), 0, st, seq_ids, seq_ok, B, W, max_batch,
                  seq_len);
}

cudaError_t launch_alloc_to_len(const int32_t* seq_ids, const int32_t* lens, int n, int relative, int32_t* seq_len,
                                int32_t* seq_npages, int32_t* page_table, uint32_t* free_bits, int max_pages,
                                int num_pages, int max_batch, int* status, cudaStream_t st) {
  return launch_k(alloc_to_len_kernel, dim3(1), dim3(32), 0, st, seq_ids, lens, n, relative, seq_len, seq_npages,
                  page_table, free_bits, max_pages, num_pages, max_batch, status);
}

cudaError_t launch_kv_fill_pages(act_t* kpool, act_t* vpool, const int32_t* page_table,
                                 const int32_t* seq_npages, int max_pages, const int32_t* seq_ids, int n,
                                 int n_layers, int num_pages, int Hkv, int hd, uint64_t seed, float scale,
                                 cudaStream_t st) {
  dim3 grid(max_pages, n_layers, n);
  return launch_k(kv_fill_kernel, grid, dim3(256), 0, st, kpool, vpool, page_table, seq_npages, max_pages, seq_ids,
                  num_pages, Hkv, hd, seed, scale);
}

}  // namespace spec
