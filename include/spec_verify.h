/*
 * spec_verify.h -- C ABI of the GB300 speculative-decoding verify round.
 *
 * One verify round, as the speculative-decoding pages describe it:
 *   - the target decoder scores W = gamma + 1 rows per sequence in ONE forward
 *     pass: row 0 is the pending token (the last committed token, whose KV is
 *     not cached yet), rows 1..gamma are the drafts
 *     (Lecture 6 "Optimizing Autoregressive Decode", sections 6.1-6.2;
 *      "Per-step cost versus accepted tokens", "What SGLang actually runs":
 *      column 0 of the verify block holds the previous bonus token);
 *   - acceptance: greedy longest matching prefix (temperature 0), or chain
 *     rejection sampling -- accept x_i while u_i * q_i(x_i) < p_i(x_i), then
 *     one draw from norm(max(0, p - q)) after a rejection, or the bonus token
 *     from p_{gamma+1} after full acceptance (Lecture 6, sections 6.2, 7.1,
 *     7.4; Leviathan Algorithm 1);
 *   - commit: the KV cache keeps the committed sequence minus its last token;
 *     after accepting n drafts the cached length becomes L + 1 + n and pages
 *     wholly beyond it return to the pool (Lecture 6, sections 6.2 and 11:
 *     rollback is a length edit of the block table).  Pages hold 64 tokens
 *     (the ninfer draft-depth sweep, "kPagedKVPageSize = 64").
 *
 * Conventions for every entry point
 *   - Tensor arguments are DEVICE pointers owned by the caller unless the
 *     comment says "host".  Row-major, no padding, int32 token ids, fp32
 *     probabilities/uniforms/logits.
 *   - All work is enqueued on `stream` (a cudaStream_t, NULL = legacy default
 *     stream) and is asynchronous; outputs are valid once the stream has
 *     synchronised.  Steps never allocate device memory.
 *   - Status return only.  Argument errors are detected on the host before any
 *     launch and return SPEC_ERR_INVALID_ARG with nothing enqueued.  Errors only
 *     the device can see (a token id out of range, an exhausted page pool, a
 *     bounded wait that ran out) set a device status word: the call that
 *     enqueued the work still returns SPEC_OK, and the next spec_sync_status()
 *     returns the code (and clears it).  Kernels that hit such an error skip the
 *     offending memory accesses, so the context stays usable.  With several
 *     errors the word keeps the first one set; within one round's preparation
 *     that is the first in batch order (per sequence: a verify length outside
 *     1..gamma+1, then a window that cannot get its pages, then a token id out
 *     of range).
 *   - A sampled (temperature > 0) round with q or u missing is an error; the
 *     library never falls back to greedy.
 *   - seq_ids of one call must be distinct and in 0..max_batch-1.  A call that
 *     breaks this is refused on the device (status word SPEC_ERR_INVALID_ARG):
 *     no KV is written and no sequence's length or pages change.  A sequence
 *     whose window cannot get its KV pages (SPEC_ERR_CAPACITY) likewise keeps
 *     its length and pages; the other sequences of the call commit normally.
 *     Outputs of refused sequences are written but carry no meaning.
 *   - spec_last_error() gives a thread-local message for the last failure.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum spec_status {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1,
  SPEC_ERR_UNSUPPORTED_DEVICE = 2, /* not an sm_103 GPU */
  SPEC_ERR_OOM = 3,                /* cudaMalloc failed at create */
  SPEC_ERR_CAPACITY = 4,           /* no free KV page / sequence longer than max_seq_len */
  SPEC_ERR_CUDA = 5,               /* a CUDA runtime call failed */
  SPEC_ERR_TIMEOUT = 6,            /* a bounded device-side wait ran out */
  SPEC_ERR_UNSUPPORTED = 7         /* a shape the kernels do not handle */
} spec_status;

/* Decoder shape and pool sizes.  d_model, n_heads*head_dim, n_kv_heads*head_dim
 * and ffn_dim must be multiples of 128 and vocab a multiple of 128; head_dim is
 * 64 or 128; n_heads a multiple of n_kv_heads with n_heads/n_kv_heads <= 8. */
typedef struct spec_config {
  int32_t n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
  float rms_eps;     /* RMSNorm epsilon inside the root */
  float rope_theta;  /* RoPE base; half-split pairs (i, i + head_dim/2) */
  int32_t page_size; /* tokens per KV page; must be 64 */
  int32_t max_batch; /* sequence slots; sequence ids are 0..max_batch-1 */
  int32_t max_width; /* rows per sequence in one forward (gamma + 1 or tree nodes), 1..16 */
  int32_t max_seq_len; /* cached tokens per sequence, <= 65536 */
  int32_t num_pages; /* KV page pool size (pages of page_size tokens, all layers) */
} spec_config;

/* Weight tensors (standard Llama layout, row-major [out, in]).
 * Matrices are bf16, norm gains fp32.  `layer` is ignored for the global ones. */
typedef enum spec_weight {
  SPEC_W_EMBED = 0,      /* [vocab, d_model] bf16 */
  SPEC_W_LM_HEAD = 1,    /* [vocab, d_model] bf16 (untied) */
  SPEC_W_FINAL_NORM = 2, /* [d_model] fp32 */
  SPEC_W_ATTN_NORM = 3,  /* [d_model] fp32 */
  SPEC_W_WQ = 4,         /* [n_heads*head_dim, d_model] bf16 */
  SPEC_W_WK = 5,         /* [n_kv_heads*head_dim, d_model] bf16 */
  SPEC_W_WV = 6,         /* [n_kv_heads*head_dim, d_model] bf16 */
  SPEC_W_WO = 7,         /* [d_model, n_heads*head_dim] bf16 */
  SPEC_W_FFN_NORM = 8,   /* [d_model] fp32 */
  SPEC_W_GATE = 9,       /* [ffn_dim, d_model] bf16 */
  SPEC_W_UP = 10,        /* [ffn_dim, d_model] bf16 */
  SPEC_W_DOWN = 11       /* [d_model, ffn_dim] bf16 */
} spec_weight;

typedef struct spec_model spec_model; /* opaque; owned by the library */

/* Create a model on the current CUDA device: validates cfg, allocates the weight
 * arena, the KV page pool, the sequence state and every workspace, all at once.
 * Weights start as zeros; load them with spec_model_set_weight.  All sequences
 * start empty.  Returns SPEC_ERR_UNSUPPORTED_DEVICE on anything but sm_103. */
spec_status spec_model_create(const spec_config* cfg, spec_model** out);

/* Free everything the model owns.  Synchronises the device first.  NULL is a no-op. */
void spec_model_destroy(spec_model* m);

/* Copy one weight tensor into the model (the library repacks it into its own
 * layout).  src may be a device or a host pointer (cudaMemcpyDefault);
 * n_elems must equal the tensor's size.  Enqueued on `stream`. */
spec_status spec_model_set_weight(spec_model* m, spec_weight which, int32_t layer,
                                  const void* src, int64_t n_elems, void* stream);

/* Empty the given sequences (host ids) and return their pages to the pool. */
spec_status spec_seq_reset(spec_model* m, int32_t n, const int32_t* seq_ids_host, void* stream);

/* Prefill: append prompt[:-1] of each sequence to its cache; the last prompt
 * token becomes the pending token, which the caller passes as row 0 of the next
 * decode/verify call.  tokens: device [B, stride] (row b holds lens_host[b]
 * tokens); seq_ids: device [B]; lens_host: HOST [B], each >= 1.  Runs the
 * target forward in windows of max_width rows per sequence. */
spec_status spec_prefill(spec_model* m, int32_t B, const int32_t* seq_ids, const int32_t* tokens,
                         int32_t stride, const int32_t* lens_host, void* stream);

/* Sampling adjustments of sampled rounds (Lecture 6 "Optimizing Autoregressive
 * Decode" section 7.3; "Per-step cost versus accepted tokens", section "Reefs"):
 * top_k, top_p are device arrays [B] (either may be NULL = off for every
 * sequence).  top_k[b] in [1, vocab) keeps sequence b's k most probable tokens
 * (0 or >= vocab: off); top_p[b] in (0, 1) then keeps the shortest top-ranked
 * prefix whose mass reaches top_p of the top-k renormalised mass (1: off).
 * Rank order: p descending, lower token index first on equal p; masses on the
 * 2^-40 grid, R_v = floor(p_v * 2^40), nucleus = the shortest prefix with summed R
 * >= ceil(fl64(top_p) * S_k); kept tokens get fl32(fl64(R_v) * fl64(1/Z)), Z =
 * their summed R.  The target p of every window row is adjusted before the
 * accept tests, the residual and the bonus draw; q must be the draft
 * distribution the drafts were drawn from -- adjusted the same way (see
 * spec_adjust_probs) for the best acceptance, though any q keeps the output law
 * equal to the adjusted p.  Ignored when temperature == 0 (the argmax is
 * unchanged).  A setting outside its range sets SPEC_ERR_INVALID_ARG in the
 * status word and leaves that sequence unadjusted.  Supported for vocab <=
 * 393216 (SPEC_ERR_INVALID_ARG otherwise). */

/* Baseline decode step (q_len = 1): one forward over the pending tokens tok[B],
 * then argmax (temperature == 0) or one draw from softmax(logits/T) with u[B]
 * (temperature > 0; u required), adjusted by top_k / top_p as above.  Writes
 * next_tok[B] and commits (L += 1). */
spec_status spec_decode_step(spec_model* m, int32_t B, const int32_t* seq_ids, const int32_t* tok,
                             float temperature, const int32_t* top_k, const float* top_p, const float* u,
                             int32_t* next_tok, void* stream);

/* Verify round.  tok [B, gamma+1]: pending token + gamma drafts.
 * temperature == 0: greedy, q and u must be NULL or are ignored.
 * temperature > 0: q [B, gamma, vocab] fp32 draft distributions (q[b, i-1] is
 * the distribution draft x_i was drawn from, over the same temperature-adjusted
 * vocabulary), u [B, gamma+1] fp32 uniforms in [0,1): u[b, i-1] drives the test
 * of x_i and u[b, gamma] the one final draw.  top_k, top_p: sampling
 * adjustments as above (NULL = off).
 * Outputs: accepted [B] = n_b; committed [B, gamma+1] = x_1..x_n then the
 * resampled or bonus token, -1 after; bonus [B] = that last token.
 * Commits L <- L + 1 + n_b and frees trailing pages.  1 <= gamma+1 <= max_width. */
spec_status spec_verify_step(spec_model* m, int32_t B, int32_t gamma, const int32_t* seq_ids,
                             const int32_t* tok, const float* q, const float* u, float temperature,
                             const int32_t* top_k, const float* top_p, int32_t* accepted, int32_t* committed,
                             int32_t* bonus, void* stream);

/* Ragged verify: each sequence verifies its own number of rows, verify_lens[b]
 * in [1, gamma+1] ("投机解码的性能收支" section 四: per-request verify lengths from
 * a planner, modes static / cap-accept / compact; the planner itself needs a
 * trained confidence head and is not here).  Sequence b accepts at most
 * verify_lens[b] - 1 drafts; u[b, verify_lens[b]-1] drives its final draw.
 *   mode SPEC_RAGGED_CAP_ACCEPT: the forward still scores gamma+1 rows per
 *     sequence (tok [B, gamma+1]); only acceptance is capped.
 *   mode SPEC_RAGGED_COMPACT: the forward scores only the real rows: tok is
 *     packed, sequence b's rows after those of sequences < b (total_rows =
 *     sum of verify_lens, passed on the host so the launch can be sized; the
 *     device checks the sum).
 * verify_lens: device [B].  q [B, gamma, V], u [B, gamma+1], committed
 * [B, gamma+1] are padded per sequence as in spec_verify_step; top_k, top_p as
 * there.  Both modes commit L + 1 + n_b and free trailing pages. */
enum { SPEC_RAGGED_CAP_ACCEPT = 1, SPEC_RAGGED_COMPACT = 2 };
spec_status spec_verify_ragged(spec_model* m, int32_t B, int32_t gamma, const int32_t* seq_ids, const int32_t* tok,
                               const int32_t* verify_lens, int32_t total_rows, int32_t mode, const float* q,
                               const float* u, float temperature, const int32_t* top_k, const float* top_p,
                               int32_t* accepted, int32_t* committed, int32_t* bonus, void* stream);

/* Greedy token-tree verify (Lecture 6 section 10.3).  tok [B, n_nodes], node 0 =
 * pending token; parent_host: HOST [n_nodes], parent[0] = -1 and
 * 0 <= parent[c] < c (BFS order).  One forward under the ancestor mask (node c
 * at position L + depth(c), KV slot L + c); the accepted path is the longest
 * root-to-node walk whose tokens equal the target argmax at their parent
 * (lowest node index among equal siblings).  Outputs: accepted [B] = path
 * length n; committed [B, n_nodes]: path tokens then the bonus token, -1 after;
 * bonus [B].  The path's KV (all layers) is moved to slots L+1..L+n, then the
 * cache is cut to L + 1 + n.  n_nodes <= max_width. */
spec_status spec_verify_tree_step(spec_model* m, int32_t B, int32_t n_nodes, const int32_t* seq_ids,
                                  const int32_t* tok, const int32_t* parent_host,
                                  int32_t* accepted, int32_t* committed, int32_t* bonus, void* stream);

/* Sampled token-tree verify (multi-draft speculative sampling).  The pages name
 * sampled tree verification (Lecture 6 section 10.3, SpecInfer; "Per-step cost
 * versus accepted tokens", section "Reefs", the non-greedy tree sampler) without
 * stating its rule; this is SpecInfer's multi-step speculative sampling, i.e.
 * recursive rejection over the children of a node: from the root, the children c
 * of the current node v are tried in node order; child c (token x) is accepted
 * when fl32(u[b, c] * q_v(x)) < p_cur(x), where p_cur is the target at v (after
 * temperature and top_k / top_p as in spec_verify_step) and, after each rejected
 * child, the normalised residual max(0, p_cur - q_v) (masses floor(r * 2^40),
 * p = fl32(fl64(R) * fl64(1 / sum R))).  After the last child of v is rejected
 * the final token is drawn from that residual; at a node without children it is
 * the bonus draw from the target at v; both by the integer inverse CDF with
 * u[b, 0].  The output follows the target distribution when the children of node v
 * were drawn i.i.d. from q[b, v] (q: device [B, n_nodes, vocab] fp32; rows of
 * leaves unused) or, with q = NULL, for any fixed set of distinct candidate tokens
 * (each child's q is then the one-hot of its own token).  u: device [B, n_nodes]
 * fp32 in [0, 1).  With parent[c] = c - 1 this is spec_verify_step's rule (tree
 * u[b, c] = chain u[b, c-1], tree u[b, 0] = chain u[b, gamma]).  Outputs and KV
 * commit as spec_verify_tree_step.  temperature > 0. */
spec_status spec_verify_tree_sampled(spec_model* m, int32_t B, int32_t n_nodes, const int32_t* seq_ids,
                                     const int32_t* tok, const int32_t* parent_host, const float* q,
                                     const float* u, float temperature, const int32_t* top_k,
                                     const float* top_p, int32_t* accepted, int32_t* committed,
                                     int32_t* bonus, void* stream);

/* Forward only: score W rows per sequence (chain, or tree if parent_host != NULL)
 * and write the window's KV, without changing any committed length.  logits_out
 * (device [B, W, vocab] fp32) may be NULL. */
spec_status spec_score(spec_model* m, int32_t B, int32_t W, const int32_t* seq_ids, const int32_t* tok,
                       const int32_t* parent_host, float* logits_out, void* stream);

/* Standalone acceptance on given probabilities (no model): p [B, gamma+1, V]
 * fp32 target probabilities (row j = distribution after row j's token),
 * q [B, gamma, V], x [B, gamma] drafts, u [B, gamma+1].  Runs the acceptance
 * kernel of spec_verify_step's sampled rounds (the same accept tests, residual
 * and integer-CDF draw across an 8-CTA cluster), reading p from memory instead
 * of deriving it from the LM head's logits; so its decisions on given p, q, u
 * are those of the model round and match a sequential CPU computation bit for
 * bit (fp32 products, integer CDF).  A row of p without mass on the 2^-40 grid
 * (not a distribution) draws token 0. */
spec_status spec_accept_probs(int32_t B, int32_t gamma, int32_t V, const float* p, const float* q,
                              const int32_t* x, const float* u, int32_t* accepted, int32_t* committed,
                              int32_t* bonus, void* stream);

/* Sampling adjustment of given probability rows (no model): p_out = top-k /
 * top-p adjustment of p (definition above spec_decode_step), row r using setting
 * r / rows_per_setting of top_k / top_p (device arrays; either may be NULL = off).
 * p, p_out: device [rows, V] fp32 probabilities (entries in [0, 1]); p_out may
 * equal p.  Rows whose setting is off, or outside its range (no status word
 * here: the row is left as it is), are copied unchanged.  For adjusting the
 * draft's q the same way as the target's p, and for spec_accept_probs on
 * adjusted rows.  rows <= 65535, V <= 393216. */
spec_status spec_adjust_probs(int32_t rows, int32_t V, const float* p, float* p_out, const int32_t* top_k,
                              const float* top_p, int32_t rows_per_setting, void* stream);

/* Standalone sampled tree acceptance on given probabilities (no model): p [B, n_nodes,
 * V] fp32 (row c = target after node c), q [B, n_nodes, V] or NULL, tok [B, n_nodes]
 * (node 0 = pending token), parent_host HOST [n_nodes], u [B, n_nodes].  Same rule and
 * outputs as spec_verify_tree_sampled, no KV commit; bit-exact by construction. */
spec_status spec_accept_tree_probs(int32_t B, int32_t n_nodes, int32_t V, const float* p, const float* q,
                                   const int32_t* tok, const int32_t* parent_host, const float* u,
                                   int32_t* accepted, int32_t* committed, int32_t* bonus, void* stream);

/* Standalone greedy acceptance on given logits [B, gamma+1, V] and drafts x [B, gamma]. */
spec_status spec_accept_greedy(int32_t B, int32_t gamma, int32_t V, const float* logits, const int32_t* x,
                               int32_t* accepted, int32_t* committed, int32_t* bonus, void* stream);

/* Greedy acceptance that allocates nothing.  The pages have no counterpart: this
 * is for callers that cannot call cudaMalloc -- code running inside another
 * framework's memory pool or a strict memory budget, or a process that must not
 * allocate once serving has started.  Same inputs and outputs as
 * spec_accept_greedy, same results; it takes the argmax of each of the
 * B*(gamma+1) logits rows in its own block (faster when V is large) and keeps
 * those argmaxes in a fixed scratch array inside the library's device memory
 * (4096 rows = 16 KB, held on every GPU that loads the library until the process
 * exits).  B*(gamma+1) > 4096 returns SPEC_ERR_INVALID_ARG.  The first call on a
 * device looks up the scratch address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  All calls share the
 * one scratch array: calls that overlap on the GPU (different streams, no
 * ordering between them) race and give undefined results.  Each row's entry is
 * rewritten before it is read, so nothing needs clearing between calls.  The
 * looked-up address is kept for the life of the process: it assumes the device's
 * primary context is never reset (cudaDeviceReset, or a context torn down and
 * created again, would leave it stale). */
spec_status spec_accept_greedy_noalloc(int32_t B, int32_t gamma, int32_t V, const float* logits,
                                       const int32_t* x, int32_t* accepted, int32_t* committed,
                                       int32_t* bonus, void* stream);

/* Synchronous host copy of the sequence state for tests: seq_len_host [n] and
 * page_table_host [n, max_pages_per_seq] (-1 = no page). */
spec_status spec_get_kv_state(spec_model* m, int32_t n, const int32_t* seq_ids_host, int32_t* seq_len_host,
                              int32_t* page_table_host);

/* Synchronous host copy of cached K and V (fp16 bits: the cache is fp16) of one
 * sequence, slots [t0, t0+n), layer `layer`: k_host and v_host are
 * [n, n_kv_heads, head_dim] uint16. */
spec_status spec_read_kv(spec_model* m, int32_t layer, int32_t seq_id, int32_t t0, int32_t n,
                         uint16_t* k_host, uint16_t* v_host);

/* Copy the last forward's logits ([rows, vocab] fp32, rows = B*W of that call)
 * to `out` (device or host).  Enqueued on `stream`. */
spec_status spec_debug_logits(spec_model* m, float* out, int64_t max_elems, void* stream);

/* Failure-path check without a fault: one device-side wait that nothing
 * completes (a fresh mbarrier phase with no arrival), bounded like every wait of
 * the library.  It runs out after budget_cycles SM clock cycles (1 ..
 * 4000000000; ~2 s at 2 GHz is the library's own budget) and records
 * SPEC_ERR_TIMEOUT in the model's status word, which the next spec_sync_status()
 * returns and clears; the context stays usable.  Enqueued on `stream`. */
spec_status spec_debug_wait_probe(spec_model* m, int64_t budget_cycles, void* stream);

/* Give sequence seq_id (host int) exactly n_tokens cached tokens whose K and V
 * are the caller's: k, v device [n_layers, n_tokens, n_kv_heads, head_dim] fp16
 * bits (the cache's format), 16-byte aligned.  The sequence is emptied first,
 * then gets pages for n_tokens slots (lowest free first) and the values copied
 * in; its length becomes n_tokens, so the next call's row 0 is the pending
 * token at position n_tokens.  Lets a test start the model and a reference
 * from one cache without a prefill.  An exhausted pool sets SPEC_ERR_CAPACITY
 * in the status word (length 0).  Synchronises `stream`. */
spec_status spec_kv_write(spec_model* m, int32_t seq_id, int32_t n_tokens, const uint16_t* k, const uint16_t* v,
                          void* stream);

/* Timing aid for long contexts: give each sequence (host ids) lens_host[b]
 * cached tokens with pseudo-random bf16 K/V (a hash of seed and position, scaled
 * by `scale`), without running the model.  Attention time does not depend on
 * the values. */
spec_status spec_kv_fill_random(spec_model* m, int32_t n, const int32_t* seq_ids_host, const int32_t* lens_host,
                                uint64_t seed, float scale, void* stream);

/* Per-kernel timing for reports.  While enabled, every weight-streaming
 * projection launch and every attention launch of a forward is bracketed by CUDA
 * events on the call's stream (this serialises those launches; use it in a
 * separate measuring pass), and no kernel prefetches the next kernel's weights
 * into L2, so every launch is timed on the bytes it moves itself.  Classes: 0 QKV, 1 O, 2 gate/up, 3 down, 4 LM head,
 * 5 attention (+ merge).  spec_read_profile synchronises the device, adds the
 * recorded durations to ms[6] and launch counts to launches[6], and its
 * algorithmic HBM bytes (weights; K/V pages read) to bytes[6], then clears the
 * record.  At most 1024 launches are recorded between two reads. */
spec_status spec_set_profiling(spec_model* m, int32_t enable);
spec_status spec_read_profile(spec_model* m, double* ms, int64_t* launches, double* bytes);

/* Synchronise `stream`, return and clear the device status word.
 * SPEC_ERR_UNSUPPORTED reported from the device means a pair of CTAs of the
 * tensor-core projection for 65+ token rows (which share one MMA across two SMs)
 * was not placed on the two SMs of one TPC and computed nothing; the model then
 * serves those row counts with single-CTA tiles from the next call on. */
spec_status spec_sync_status(spec_model* m, void* stream);

/* Pages per sequence in the page table (ceil(max_seq_len / page_size)). */
int32_t spec_max_pages_per_seq(const spec_model* m);

/* Number of kernel launches the last forward/round enqueued (for reports). */
int32_t spec_last_launch_count(const spec_model* m);

/* Message for the last error on this thread ("" if none). */
const char* spec_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
