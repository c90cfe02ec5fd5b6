// Host-side launchers shared between the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace spec {

// Launch with programmatic stream serialization (PDL) so a kernel's prologue
// (weight prefetch) overlaps the tail of the kernel before it.
extern bool g_use_pdl;

// Message for spec_last_error() (thread-local), for entry points outside api.cu.
void record_error(const char* msg);

// Fused-epilogue projection (gemm.cu).  Y = X W^T over M rows; W: [N, K] fp16 with
// a per-row scale (tensor map box {64, 128}), X: [M_alloc, K] fp16 (box {64, BM}).
// With split-K the splits of a tile run as one thread-block cluster and reduce
// their partial tiles through distributed shared memory before the epilogue:
enum { kEpiQKV = 0, kEpiSwiGLU = 1, kEpiResid = 2, kEpiLogits = 3 };
struct EpiParams {
  int M, N, K;
  int kb_total, kb_per_split, splits;  // kb_* filled by the launcher
  const float* rscale;                 // [N] 2^-e of each weight row's fp16 encoding
  // row scale of a normalised input (ssq_in = null: scale 1)
  const float* ssq_in;                 // [ssq_tiles][ssq_stride] partial sums of r^2
  int ssq_tiles, ssq_stride;
  float inv_d, eps;
  // kEpiQKV: RoPE + q out + paged K/V write
  int Hq, Hkv, hd;
  const int32_t* row_pos;
  const int32_t* row_slot;
  const float* rope_cos;
  const float* rope_sin;
  __half* q_out;
  __half* kpool;                       // this layer's base
  __half* vpool;
  // kEpiSwiGLU
  __half* act;
  int ffn;
  // kEpiResid: resid += y, xn = fp16(resid * g_next), ssq_out partial sums
  float* resid;
  const float* g_next;
  __half* xn;
  float* ssq_out;
  int d;
  // kEpiLogits: logits and per-128-column (max, sum exp((l-max)/T), argmax) of each row
  float* logits;
  float inv_temp;
  float* tstat_max;
  float* tstat_sum;                    // null: greedy (no sum)
  int32_t* tstat_arg;
  int tstat_stride;
  // Weights of the next projection, brought into L2 by each CTA's producer once
  // its own weight stream is issued (HBM idles while the grid drains and the next
  // kernel starts); split evenly over the CTAs.  Null / 0: none.
  const void* l2_next;
  unsigned long long l2_next_bytes;  // multiple of 16
  int tok_tile;                      // token rows per tile (pair kernel; 0: the kernel's tile)
  int tok_chunk;                     // token rows per epilogue chunk (pair kernel)
  int sm_count;
  // Set by the launcher: release the next kernel (programmatic dependent launch) only
  // as each CTA finishes, for grids of more than one wave.  Released early, the next
  // grid's clusters are placed piecemeal on the slots this grid's last wave frees and
  // part of it ends up in a second wave.
  int late_dependents;
  int* status;
};
cudaError_t launch_gemm_epi(int epi, const CUtensorMap* tmW, const CUtensorMap* tmX, int BM, EpiParams p,
                            cudaStream_t st);

// Choose split-K for an N x K projection over M rows so that the grid fills the GPU.
int choose_splits(int N, int K, int M, int BM, int sm_count, int max_splits);
int choose_bm(int M);
// CTA-pair tcgen05 kernel (BM = kPairBM; every N a multiple of 256): whether it
// serves M token rows, and its token tile (rows per tile, at most 256, a multiple
// of 16; its X tensor map has boxes of pair_tile_rows(M) / 2 rows).
constexpr int kPairBM = 256;
bool pair_rows(int M);
int pair_tile_rows(int M);

// --- elementwise (elementwise.cu): resid = E[tok]; xn = fp16(E[tok] * g); ssq partials
cudaError_t launch_embed(const int32_t* tok, int M, const __nv_bfloat16* embed, const float* gain, int d, int vocab,
                         float* resid, __half* xn, float* ssq_out, int ssq_stride, int* status, cudaStream_t st);
// bf16 rows -> fp16 * 2^e rows, in place; rscale[row] = 2^-e
cudaError_t launch_encode_rows(uint16_t* w, int K, int n_rows, int block, int block_stride, int row0, float* rscale,
                               cudaStream_t st);

// --- attention (attention.cu)
struct AttnParams {
  const __half* q;             // [M, Hq*hd] rotated queries
  const int32_t* page_table;   // [max_batch, max_pages]
  const int32_t* seq_ids;      // [B]
  const int32_t* seq_start;    // [B] cached length L at round start
  const int32_t* seq_wlen;     // [B] window rows of sequence b
  const int32_t* seq_rowoff;   // [B] first flat row of sequence b
  const int32_t* seq_order;    // [B] batch index of the z-th CTA group (longest cache first)
  int max_pages, max_batch;
  int B, W, Hq, Hkv, hd;       // W: the widest window of the call
  int layer_row0;              // first TMA row of this layer in the KV pool maps
  int sm_count;                // picks the cluster size (1 to 16 CTAs per sequence and kv head)
  int kv_len_hint;             // upper bound of L + W over the batch (launch shape only)
  uint32_t anc[16];            // ancestor masks of the window rows (bit i: row i visible)
  // Weights of the projections that follow, brought into L2 once the QKV
  // projection is done (HBM is otherwise idle while a short-context attention
  // runs); split evenly over the CTAs.  Null / 0: none.
  const void* l2_next[2];
  unsigned long long l2_next_bytes[2];  // multiples of 16
  int late_trigger;            // set by the launcher: release the successor after the queries arrive
  __half* out;                 // [M, Hq*hd]
  int* status;
};
cudaError_t launch_attention(const CUtensorMap* tmK, const CUtensorMap* tmV, const AttnParams& p, cudaStream_t st);

// --- sequence state, acceptance and commit (accept.cu)
struct PrepareParams {
  const int32_t* seq_ids;   // [B]
  int B, W;                 // W: rows of every sequence, or the widest when `wlen` is given
  const int32_t* wlen;      // [B] rows per sequence (device), or null: W each
  int total_rows;           // sum of the rows (checked on the device when wlen is given)
  int32_t* seq_wlen;        // [B] out: rows of sequence b
  int32_t* seq_rowoff;      // [B] out: first flat row of sequence b
  int32_t* seq_len;         // [max_batch]
  int32_t* seq_npages;      // [max_batch]
  int32_t* page_table;      // [max_batch, max_pages]
  uint32_t* free_bits;      // [ceil(num_pages/32)], bit set = free
  int num_pages, max_pages, max_seq_len, max_batch;
  int depth[16];            // position offset of window row j
  int32_t* row_pos;         // [B*W]
  int32_t* row_slot;        // [B*W] physical slot (page*64 + off) or -1
  int32_t* seq_start;       // [B]
  int32_t* seq_ok;          // [B] out: 1 = the window got its pages and may commit
  int32_t* seq_order;       // [B] out: batch indices by cached length, longest first
  const int32_t* tok;       // [B*W] token ids to validate
  int vocab;
  int* status;
};
cudaError_t launch_prepare(const PrepareParams& p, cudaStream_t st);

enum class PSource { kLogits = 0, kProbs = 1 };

// Standalone greedy acceptance on given logits (no model, no commit).
struct AcceptParams {
  int B, gamma, V;
  const float* rows;          // [B*W, V] logits
  const int32_t* tok;         // [B, gamma] drafts
  const int32_t* row_argmax;  // [B*W] argmax of each row, or null: taken inside the kernel
  int32_t* accepted;          // [B]
  int32_t* committed;         // [B, W]
  int32_t* bonus;             // [B]
};
cudaError_t launch_row_stats(const float* rows, int n_rows, int V, float inv_temp, bool sampled, int32_t* argmax,
                             float* row_max, float* row_sum, cudaStream_t st);
cudaError_t launch_accept_greedy(const AcceptParams& p, cudaStream_t st);

// Acceptance of a model round from the LM head's per-tile statistics.
constexpr int kDrawCluster = 8;
constexpr int kMaxDrawCluster = 16;
struct SelRow;
struct RoundAcceptParams {
  int B, gamma, V;           // gamma: the widest window - 1 (stride of q, u, committed)
  const int32_t* seq_wlen;   // [B] window rows of sequence b (null: gamma + 1 each)
  const int32_t* seq_rowoff; // [B] first flat row of sequence b (null: b * (gamma + 1))
  const int32_t* cap;        // [B] acceptance cap (verify length) or null
  float inv_temp;
  const float* logits;       // [B*W, V]
  int n_tiles;               // V / 128
  const float* tstat_max;    // [n_tiles][tstat_stride]
  const float* tstat_sum;
  const int32_t* tstat_arg;
  int tstat_stride;
  const float* probs;        // [B*W, V] given target probabilities (PSource::kProbs)
  const float* q;            // [B, gamma, V] (sampled)
  const int32_t* tok;        // [rows] window tokens, sequence b at seq_rowoff[b]
  const int32_t* x;          // [B, gamma] drafts (standalone) or null: x_i = window row i
  const float* u;            // [B, gamma+1] (sampled)
  int32_t* accepted;
  int32_t* committed;        // [B, W]
  int32_t* bonus;
  const int32_t* seq_ids;    // null: no commit
  const int32_t* seq_ok;     // [B] from the prepare kernel: 0 = leave the sequence as it was
  int32_t* seq_len;
  int32_t* seq_npages;
  int32_t* page_table;
  uint32_t* free_bits;
  int max_pages, max_batch;
  int* status;
  // sampling adjustments (null: none): per window row, from the selection kernel
  const SelRow* sel;
  const float* sel_max;
  const float* sel_z;
};
cudaError_t launch_accept_round(const RoundAcceptParams& p, bool sampled, cudaStream_t st);
// Sampled acceptance of given probabilities (p.probs, p.x; no commit) by the same kernel.
cudaError_t launch_accept_round_probs(const RoundAcceptParams& p, cudaStream_t st);

// ---------------------------------------------------------------- top-k / top-p
constexpr int kSelCluster = 8;             // CTAs per probability row
constexpr int kSelMaxSlice = 48 * 1024;    // probability keys per CTA (shared memory)
struct SelectParams {
  int V;
  const int32_t* top_k;      // [sets] 0 (or >= V) = off
  const float* top_p;        // [sets] 1 = off
  // probabilities in, adjusted probabilities out (standalone): row r uses set r / rows_per_set
  const float* p_in;
  float* p_out;
  int rows_per_set;
  // model rounds: logits + LM-head tile statistics in, one SelRow per window row out
  const float* logits;
  const float* tstat_max;
  const float* tstat_sum;
  int n_tiles, tstat_stride;
  float inv_temp;
  const int32_t* seq_wlen;   // [B]
  const int32_t* seq_rowoff; // [B]
  SelRow* sel;               // [rows]
  float* row_max;            // [rows] merged softmax statistics the acceptance reuses
  float* row_z;
  int* status;
};
int select_max_vocab();
// kProbs: grid rows = n_rows; kLogits: n_rows_or_wmax = widest window, B sequences.
cudaError_t launch_select(const SelectParams& p, PSource src, int n_rows_or_wmax, int B, cudaStream_t st);

struct TreeParams {
  int B, N, V;
  int parent[16];
  const int32_t* tok;        // [B, N]
  RoundAcceptParams stats;   // tile statistics of the B*N node rows (greedy)
  int32_t* accepted;
  int32_t* committed;        // [B, N]
  int32_t* bonus;
  const int32_t* seq_ids;
  const int32_t* seq_ok;     // [B] from the prepare kernel: 0 = no KV move, no commit
  int32_t* seq_len;
  int32_t* seq_npages;
  int32_t* page_table;
  uint32_t* free_bits;
  int max_pages, max_batch;
  __half* kpool;
  __half* vpool;
  int n_layers, num_pages, Hkv, hd;
  int* status;
  // sampled trees: q [B, N, V] (children of node v drawn i.i.d. from q[b, v]; null:
  // deterministic candidates), u [B, N] (u[b, c] tests child c, u[b, 0] the final
  // draw), probs [B, N, V] given probabilities (standalone; null: from the logits),
  // path [B, N] accepted node ids for the commit (null: no commit)
  const float* q;
  const float* u;
  const float* probs;
  int32_t* path;
};
cudaError_t launch_accept_tree(const TreeParams& p, cudaStream_t st);
// Sampled tree: the walk (cluster per sequence), then, if p.path and p.seq_ids, the KV commit.
cudaError_t launch_accept_tree_sampled(const TreeParams& p, cudaStream_t st);

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
// One bounded wait that nothing completes: records SPEC_ERR_TIMEOUT after `budget` cycles.
cudaError_t launch_wait_probe(int* status, unsigned long long budget, cudaStream_t st);
cudaError_t launch_commit_all(const int32_t* seq_ids, const int32_t* seq_ok, int B, int W, int max_batch,
                              int32_t* seq_len, cudaStream_t st);
// Sequence seq_id gets pages for n slots (lowest free first; it must be empty) and
// the given K/V ([n_layers][n][Hkv][hd] fp16 each) copied into them; length n.
cudaError_t launch_kv_write(__half* kpool, __half* vpool, const int32_t* page_table, int max_pages, int seq_id, int n,
                            const __half* k, const __half* v, int n_layers, int num_pages, int Hkv, int hd,
                            cudaStream_t st);
cudaError_t launch_alloc_to_len(const int32_t* seq_ids, const int32_t* lens, int n, int relative, int32_t* seq_len,
                                int32_t* seq_npages, int32_t* page_table, uint32_t* free_bits, int max_pages,
                                int num_pages, int max_batch, int* status, cudaStream_t st);
cudaError_t launch_kv_fill_pages(__half* kpool, __half* vpool, const int32_t* page_table,
                                 const int32_t* seq_npages, int max_pages, const int32_t* seq_ids, int n,
                                 int n_layers, int num_pages, int Hkv, int hd, uint64_t seed, float scale,
                                 cudaStream_t st);
cudaError_t launch_gather_tokens(const int32_t* tokens, int stride, const int32_t* perm, int k, int col0, int W,
                                 int32_t* out, const int32_t* seq_ids, int32_t* ids_out, cudaStream_t st);
cudaError_t launch_init_state(int32_t* seq_len, int32_t* seq_npages, int32_t* page_table, uint32_t* free_bits,
                              int max_batch, int max_pages, int num_pages, cudaStream_t st);

}  // namespace spec
