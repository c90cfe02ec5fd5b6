// Host-side launchers shared between the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace spec {

// Launch with programmatic stream serialization (PDL) so a kernel's prologue
// (weight prefetch) overlaps the tail of the kernel before it.
extern bool g_use_pdl;

// Message for spec_last_error() (thread-local), for entry points outside api.cu.
void record_error(const char* msg);

// Y_partial[split][m][n] = sum_{k in split} X[m][k] * W[n][k]
// tmW: weight map, box {64, 128}; tmX: activation map, box {64, BM}; BM in {8,16,32,64}.
// splits == 1 writes the final result (out[m*ldo + n]).
cudaError_t launch_gemm(const CUtensorMap* tmW, const CUtensorMap* tmX, int BM, int N, int K, int M, int splits,
                        float* out, long long split_stride, int ldo, int* status, cudaStream_t st);

// Choose split-K for an N x K projection over M rows so that the grid fills the GPU.
int choose_splits(int N, int K, int M, int BM, int sm_count, int max_splits);
int choose_bm(int M);

// --- elementwise (elementwise.cu)
cudaError_t launch_embed_norm(const int32_t* tok, int M, const __nv_bfloat16* embed, const float* gain, int d,
                              int vocab, float eps, float* resid, __nv_bfloat16* xn, int* status, cudaStream_t st);
cudaError_t launch_qkv_epilogue(const float* part, int splits, long long split_stride, int M, int n_heads,
                                int n_kv, int hd, const int32_t* row_pos, const int32_t* row_slot,
                                const float* rope_cos, const float* rope_sin, __nv_bfloat16* q_out,
                                __nv_bfloat16* kpool_layer, __nv_bfloat16* vpool_layer, cudaStream_t st);
cudaError_t launch_resid_norm(const float* part, int splits, long long split_stride, int M, int d, const float* gain,
                              float eps, float* resid, __nv_bfloat16* xn, cudaStream_t st);
cudaError_t launch_swiglu(const float* part, int splits, long long split_stride, int M, int ffn,
                          __nv_bfloat16* act, cudaStream_t st);

// --- attention (attention.cu)
struct AttnParams {
  const __nv_bfloat16* q;      // [M, Hq*hd] rotated queries
  const int32_t* page_table;   // [max_batch, max_pages]
  const int32_t* seq_ids;      // [B]
  const int32_t* seq_start;    // [B] cached length L at round start
  int max_pages, max_batch;
  int B, W, Hq, Hkv, hd;
  int layer_row0;              // first TMA row of this layer in the KV pool maps
  int pages_per_split, n_splits;
  uint32_t anc[16];            // ancestor masks of the window rows (bit i: row i visible)
  float* part_acc;             // [M*Hq, n_splits, hd]
  float* part_ml;              // [M*Hq, n_splits, 2]
  int* status;
};
cudaError_t launch_attention(const CUtensorMap* tmK, const CUtensorMap* tmV, const AttnParams& p, cudaStream_t st);
cudaError_t launch_attn_merge(const float* part_acc, const float* part_ml, int M, int Hq, int hd, int n_splits,
                              __nv_bfloat16* out, cudaStream_t st);

// --- sequence state, acceptance and commit (accept.cu)
struct PrepareParams {
  const int32_t* seq_ids;   // [B]
  int B, W;
  int32_t* seq_len;         // [max_batch]
  int32_t* seq_npages;      // [max_batch]
  int32_t* page_table;      // [max_batch, max_pages]
  uint32_t* free_bits;      // [ceil(num_pages/32)], bit set = free
  int num_pages, max_pages, max_seq_len, max_batch;
  int depth[16];            // position offset of window row j
  int32_t* row_pos;         // [B*W]
  int32_t* row_slot;        // [B*W] physical slot (page*64 + off) or -1
  int32_t* seq_start;       // [B]
  const int32_t* tok;       // [B*W] token ids to validate
  int vocab;
  int* status;
};
cudaError_t launch_prepare(const PrepareParams& p, cudaStream_t st);

enum class PSource { kLogits = 0, kProbs = 1 };

struct AcceptParams {
  int B, gamma, V;
  float inv_temp;           // 1/T for sampled rounds
  const float* rows;        // [B*W, V] logits or probabilities
  const float* q;           // [B, gamma, V] (sampled) or null
  const int32_t* tok;       // [B, W] window tokens (x_i = tok[b, i]) -- or drafts when x_stride == gamma
  int tok_stride, tok_offset;
  const float* u;           // [B, W] (sampled) or null
  const int32_t* row_argmax;  // [B*W] (greedy)
  const float* row_max;     // [B*W] (sampled, logits)
  const float* row_sum;     // [B*W] (sampled, logits)
  int32_t* accepted;        // [B]
  int32_t* committed;       // [B, W]
  int32_t* bonus;           // [B]
  // commit (null seq_ids = no commit)
  const int32_t* seq_ids;
  int32_t* seq_len;
  int32_t* seq_npages;
  int32_t* page_table;
  uint32_t* free_bits;
  int max_pages, max_batch;
  int* status;
};
cudaError_t launch_row_stats(const float* rows, int n_rows, int V, float inv_temp, bool sampled, int32_t* argmax,
                             float* row_max, float* row_sum, cudaStream_t st);
cudaError_t launch_accept_chain(const AcceptParams& p, bool sampled, PSource src, cudaStream_t st);

struct TreeParams {
  int B, N, V;
  int parent[16];
  const int32_t* tok;        // [B, N]
  const int32_t* row_argmax; // [B*N]
  int32_t* accepted;
  int32_t* committed;        // [B, N]
  int32_t* bonus;
  const int32_t* seq_ids;
  int32_t* seq_len;
  int32_t* seq_npages;
  int32_t* page_table;
  uint32_t* free_bits;
  int max_pages, max_batch;
  __nv_bfloat16* kpool;
  __nv_bfloat16* vpool;
  int n_layers, num_pages, Hkv, hd;
  int* status;
};
cudaError_t launch_accept_tree(const TreeParams& p, cudaStream_t st);

struct ResetParams {
  const int32_t* seq_ids;
  int n;
  int32_t* seq_len;
  int32_t* seq_npages;
  int32_t* page_table;
  uint32_t* free_bits;
  int max_pages;
};
cudaError_t launch_seq_reset(const ResetParams& p, cudaStream_t st);
cudaError_t launch_commit_all(const int32_t* seq_ids, int B, int W, int max_batch, int32_t* seq_len,
                              cudaStream_t st);
cudaError_t launch_alloc_to_len(const int32_t* seq_ids, const int32_t* lens, int n, int relative, int32_t* seq_len,
                                int32_t* seq_npages, int32_t* page_table, uint32_t* free_bits, int max_pages,
                                int num_pages, int max_batch, int* status, cudaStream_t st);
cudaError_t launch_kv_fill_pages(__nv_bfloat16* kpool, __nv_bfloat16* vpool, const int32_t* page_table,
                                 const int32_t* seq_npages, int max_pages, const int32_t* seq_ids, int n,
                                 int n_layers, int num_pages, int Hkv, int hd, uint64_t seed, float scale,
                                 cudaStream_t st);
cudaError_t launch_gather_tokens(const int32_t* tokens, int stride, const int32_t* perm, int k, int col0, int W,
                                 int32_t* out, const int32_t* seq_ids, int32_t* ids_out, cudaStream_t st);
cudaError_t launch_init_state(int32_t* seq_len, int32_t* seq_npages, int32_t* page_table, uint32_t* free_bits,
                              int max_batch, int max_pages, int num_pages, cudaStream_t st);

}  // namespace spec
