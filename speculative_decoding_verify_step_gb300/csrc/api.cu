// C ABI of the verify-round library: model arena, tensor maps, the forward
// schedule, and every entry point declared in spec_verify.h.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "sampling.cuh"

namespace spec {
bool g_use_pdl = true;
int g_launch_count = 0;
void record_error(const char* msg);
}  // namespace spec

using namespace spec;

namespace {

thread_local std::string g_err;

spec_status fail(spec_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

}  // namespace

void spec::record_error(const char* msg) { g_err = msg; }

namespace {

#define CUDA_TRY(expr)                                                                          \
  do {                                                                                          \
    cudaError_t e_ = (expr);                                                                    \
    if (e_ != cudaSuccess)                                                                      \
      return fail(SPEC_ERR_CUDA, "%s failed: %s (%s:%d)", #expr, cudaGetErrorString(e_), __FILE__, __LINE__); \
  } while (0)

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D fp16 map over a row-major [outer, inner] array, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kPairBoxes = 16;
constexpr int kNumBM = 4;
constexpr int kBMs[kNumBM] = {8, 16, 64, 128};
int bm_index(int bm) {
  for (int i = 0; i < kNumBM; ++i)
    if (kBMs[i] == bm) return i;
  return 0;
}

}  // namespace

struct spec_model {
  spec_config cfg{};
  int device = 0, sm_count = 0;
  int max_pages = 0, M_max = 0, qkv_n = 0, q_dim = 0, kv_dim = 0;
  std::vector<void*> allocs;
  // weights
  __nv_bfloat16* embed = nullptr;  // gathered, kept bf16
  act_t* lm_head = nullptr;        // projections: fp16 re-encoding with a per-row scale
  float* rs_lm = nullptr;
  float* final_norm = nullptr;
  struct Layer {
    act_t *wqkv, *wo, *wgu, *wdown;
    float *rs_qkv, *rs_o, *rs_gu, *rs_down;
    float *attn_norm, *ffn_norm;
    CUtensorMap tm_qkv, tm_o, tm_gu, tm_down;
  };
  std::vector<Layer> layers;
  CUtensorMap tm_lm;
  // KV pool: [layer][page][kv head][64][head_dim] for K and for V
  act_t *kpool = nullptr, *vpool = nullptr;
  CUtensorMap tm_k, tm_v;
  // sequence state
  int32_t *seq_len = nullptr, *seq_npages = nullptr, *page_table = nullptr;
  uint32_t* free_bits = nullptr;
  int* status = nullptr;
  std::vector<long long> host_len_bound;
  // workspaces
  float* resid = nullptr;
  act_t *xn = nullptr, *qrot = nullptr, *attn_out = nullptr, *act = nullptr;
  float *ssq_a = nullptr, *ssq_b = nullptr;  // [d/128][M_max] partial sums of r^2
  float* logits = nullptr;
  float *tstat_max = nullptr, *tstat_sum = nullptr;  // [V/128][M_max] LM-head tile statistics
  int32_t* tstat_arg = nullptr;
  SelRow* sel = nullptr;                  // [M_max] top-k / top-p kept set of each window row
  int32_t* tree_path = nullptr;           // [M_max] accepted node ids of a sampled tree round
  float *sel_max = nullptr, *sel_z = nullptr;
  int32_t *row_pos = nullptr, *row_slot = nullptr, *seq_start = nullptr;
  int32_t *seq_wlen = nullptr, *seq_rowoff = nullptr;  // per-call window layout (prepare kernel)
  int32_t* seq_ok = nullptr;  // per-call: 1 = the window got its pages and may commit
  int32_t* seq_order = nullptr;  // per-call: batch indices by cached length, longest first
  float *rope_cos = nullptr, *rope_sin = nullptr;
  int32_t *scratch_ids = nullptr, *scratch_ids2 = nullptr, *scratch_tok = nullptr, *scratch_lens = nullptr;
  int32_t *scratch_acc = nullptr, *scratch_bonus = nullptr;
  CUtensorMap tm_xn[kNumBM], tm_attn[kNumBM], tm_act[kNumBM];
  // CTA-pair kernel: boxes of 8, 16, .., 128 token rows (half a token tile)
  CUtensorMap tm_xn2[kPairBoxes], tm_attn2[kPairBoxes], tm_act2[kPairBoxes];
  bool pair_ok = false;  // every projection's N is a multiple of 256 (the pair's weight rows)
  int M_alloc = 0;  // rows of the activation buffers (>= 256 for the widest token tile)
  int last_rows = 0, last_launches = 0;
  // profiling: event pairs around projection / attention launches
  bool profiling = false;
  std::vector<cudaEvent_t> prof_ev;
  struct ProfRec {
    int cls;
    double bytes;
  };
  std::vector<ProfRec> prof_rec;
};

namespace {

spec_status alloc(spec_model* m, void** p, size_t bytes) {
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) return fail(SPEC_ERR_OOM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
  m->allocs.push_back(*p);
  CUDA_TRY(cudaMemset(*p, 0, bytes));
  return SPEC_OK;
}

template <typename T>
spec_status alloc_t(spec_model* m, T** p, size_t n) {
  return alloc(m, reinterpret_cast<void**>(p), n * sizeof(T));
}

spec_status validate_cfg(const spec_config& c) {
  if (c.n_layers < 1 || c.d_model < 128 || c.n_heads < 1 || c.n_kv_heads < 1 || c.vocab < 128)
    return fail(SPEC_ERR_INVALID_ARG, "non-positive model dimension");
  if (c.head_dim != 64 && c.head_dim != 128) return fail(SPEC_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (c.n_heads % c.n_kv_heads) return fail(SPEC_ERR_INVALID_ARG, "n_heads must be a multiple of n_kv_heads");
  if (c.n_heads / c.n_kv_heads > 8) return fail(SPEC_ERR_UNSUPPORTED, "group size above 8");
  if (c.d_model % 128 || (c.n_heads * c.head_dim) % 128 || (c.n_kv_heads * c.head_dim) % 64 || c.ffn_dim % 128 ||
      c.vocab % 128)
    return fail(SPEC_ERR_UNSUPPORTED, "projection widths must be multiples of 128");
  if (((c.n_heads + 2 * c.n_kv_heads) * c.head_dim) % 128)
    return fail(SPEC_ERR_UNSUPPORTED, "fused QKV width must be a multiple of 128");
  if (c.page_size != kPage) return fail(SPEC_ERR_UNSUPPORTED, "page_size must be 64");
  if (c.max_batch < 1 || c.max_batch > 4096) return fail(SPEC_ERR_INVALID_ARG, "max_batch out of range");
  if (c.max_width < 1 || c.max_width > kMaxWidth) return fail(SPEC_ERR_INVALID_ARG, "max_width must be 1..16");
  if (c.max_width * (c.n_heads / c.n_kv_heads) > 64)
    return fail(SPEC_ERR_UNSUPPORTED, "max_width * group size must be <= 64");
  if (c.max_seq_len < 1 || c.max_seq_len > 65536) return fail(SPEC_ERR_INVALID_ARG, "max_seq_len must be 1..65536");
  if (c.num_pages < 1) return fail(SPEC_ERR_INVALID_ARG, "num_pages must be positive");
  if (!(c.rms_eps >= 0.f) || !(c.rope_theta > 0.f)) return fail(SPEC_ERR_INVALID_ARG, "bad rms_eps / rope_theta");
  return SPEC_OK;
}

// Bytes prefetched into L2 around a latency-bound attention launch (it runs ~9 us;
// the prefetch also overlaps the O projection's start), after the QKV projection
// has prefetched the O projection's weights: the start of gate/up.  Measured at
// B = 1, width 5: 2.79 ms per round with O from the QKV projection and 45 MB here
// (30-60 MB within 0.2%), 2.85 ms with 90 MB here (O and gate/up) and nothing from
// the QKV projection, whose own weights arrive under the previous kernels.
constexpr double kAttnL2Budget = 45e6;
// Bytes of the next projection's weights prefetched into L2 at the end of each
// projection's weight stream (HBM idles while its grid drains, ~2-3 us).  Only
// while the projections are weight streams (mma.sync tiles, <= 16 token rows; measured: neutral
// to slightly negative on the tensor-core path).
constexpr double kProjL2Budget = 16e6;

long long max_len_bound(const spec_model* m) {
  long long b = 0;
  for (long long v : m->host_len_bound) b = std::max(b, v);
  return b;
}

// One target forward over B sequences x W rows.  depth[j]: position offset of row j;
// anc[j]: rows visible to row j inside the window.
template <typename F>
cudaError_t profiled(spec_model* m, int cls, double bytes, cudaStream_t st, F&& launch);

// One target forward over B sequences x W rows.  depth[j]: position offset of row j;
// anc[j]: rows visible to row j inside the window.  want_logits: run the LM head
// (with per-tile softmax statistics at temperature 1/inv_temp when `sampled`).
spec_status forward(spec_model* m, int B, int W, const int32_t* seq_ids, const int32_t* tok, const int* depth,
                    const uint32_t* anc, bool want_logits, bool sampled, float inv_temp, cudaStream_t st,
                    const int32_t* wlen = nullptr, int total_rows = -1) {
  const spec_config& c = m->cfg;
  const int M = wlen ? total_rows : B * W;  // flat rows (ragged: the caller's total)
  const int d = c.d_model, hd = c.head_dim;
  const int Hq = c.n_heads, Hkv = c.n_kv_heads, F = c.ffn_dim;

  PrepareParams pp{};
  pp.seq_ids = seq_ids;
  pp.B = B;
  pp.W = W;
  pp.wlen = wlen;
  pp.total_rows = M;
  pp.seq_wlen = m->seq_wlen;
  pp.seq_rowoff = m->seq_rowoff;
  pp.seq_len = m->seq_len;
  pp.seq_npages = m->seq_npages;
  pp.page_table = m->page_table;
  pp.free_bits = m->free_bits;
  pp.num_pages = c.num_pages;
  pp.max_pages = m->max_pages;
  pp.max_seq_len = c.max_seq_len;
  pp.max_batch = c.max_batch;
  for (int j = 0; j < 16; ++j) pp.depth[j] = j < W ? depth[j] : 0;
  pp.row_pos = m->row_pos;
  pp.row_slot = m->row_slot;
  pp.seq_start = m->seq_start;
  pp.seq_ok = m->seq_ok;
  pp.seq_order = m->seq_order;
  pp.tok = tok;
  pp.vocab = c.vocab;
  pp.status = m->status;
  CUDA_TRY(launch_prepare(pp, st));
  CUDA_TRY(launch_embed(tok, M, m->embed, m->layers[0].attn_norm, d, c.vocab, m->resid, m->xn, m->ssq_a, m->M_max,
                        m->status, st));

  const bool pair = m->pair_ok && pair_rows(M);
  const int BM = pair ? kPairBM : choose_bm(M);
  const int bi = bm_index(BM);
  const int pbox = pair ? pair_tile_rows(M) / 16 - 1 : 0;
  const CUtensorMap* tmx_xn = pair ? &m->tm_xn2[pbox] : &m->tm_xn[bi];
  const CUtensorMap* tmx_attn = pair ? &m->tm_attn2[pbox] : &m->tm_attn[bi];
  const CUtensorMap* tmx_act = pair ? &m->tm_act2[pbox] : &m->tm_act[bi];
  auto splits_for = [&](int N, int K) {
    return choose_splits(N, K, M, BM, m->sm_count, 16);
  };
  EpiParams base{};
  base.M = M;
  base.ssq_tiles = d / 128;
  base.ssq_stride = m->M_max;
  base.inv_d = 1.f / d;
  base.eps = c.rms_eps;
  base.status = m->status;
  base.sm_count = m->sm_count;

  AttnParams ap{};
  ap.q = m->qrot;
  ap.page_table = m->page_table;
  ap.seq_ids = seq_ids;
  ap.seq_start = m->seq_start;
  ap.seq_wlen = m->seq_wlen;
  ap.seq_rowoff = m->seq_rowoff;
  ap.seq_order = m->seq_order;
  ap.max_pages = m->max_pages;
  ap.max_batch = c.max_batch;
  ap.B = B;
  ap.W = W;
  ap.Hq = Hq;
  ap.Hkv = Hkv;
  ap.hd = hd;
  for (int j = 0; j < 16; ++j) ap.anc[j] = j < W ? anc[j] : 0u;
  ap.out = m->attn_out;
  ap.sm_count = m->sm_count;
  ap.kv_len_hint = (int)std::min<long long>(max_len_bound(m) + W, c.max_seq_len);
  ap.status = m->status;

  const long long layer_elems = (long long)c.num_pages * Hkv * kPage * hd;
  const double wb_qkv = 2.0 * m->qkv_n * d, wb_o = 2.0 * d * m->q_dim, wb_gu = 4.0 * F * d, wb_dn = 2.0 * d * F;
  // K/V bytes of one attention launch: the host-side bound on the cached lengths
  const long long bound = std::min<long long>(max_len_bound(m) + W, c.max_seq_len);
  const double kv_bytes = 2.0 * 2.0 * hd * Hkv * (double)B * (double)bound;
  // While a short-context attention runs, HBM has room for about kAttnL2Budget
  // bytes beyond the attention's own K/V: that much of the O projection's and
  // then the gate/up projection's weights is prefetched into L2 (none once the
  // K/V reads alone fill the attention's time).
  // While per-kernel profiling is on, no kernel prefetches another's weights: each
  // launch is then timed on the bytes it moves itself.
  const bool prefetch = !m->profiling;
  const double proj_pf = prefetch && BM <= 16 ? kProjL2Budget : 0.0;
  // The QKV projection (mma.sync tiles) prefetches the O projection's weights; the
  // attention, what is left of them and then the start of gate/up.
  const unsigned long long q_o = prefetch && BM <= 16 ? (unsigned long long)wb_o & ~15ull : 0ull;
  const double pf = prefetch ? std::max(0.0, kAttnL2Budget - kv_bytes) : 0.0;
  const unsigned long long pf_o = (unsigned long long)std::min(pf, wb_o - (double)q_o) & ~15ull;
  const unsigned long long pf_gu = (unsigned long long)std::max(0.0, std::min(pf - (double)pf_o, wb_gu)) & ~15ull;
  for (int l = 0; l < c.n_layers; ++l) {
    auto& Ly = m->layers[l];
    ap.l2_next[0] = reinterpret_cast<const char*>(Ly.wo) + q_o;
    ap.l2_next_bytes[0] = pf_o;
    ap.l2_next[1] = Ly.wgu;
    ap.l2_next_bytes[1] = pf_gu;
    {
      EpiParams e = base;
      e.N = m->qkv_n;
      e.K = d;
      e.rscale = Ly.rs_qkv;
      e.splits = splits_for(e.N, e.K);
      e.ssq_in = m->ssq_a;
      e.Hq = Hq;
      e.Hkv = Hkv;
      e.hd = hd;
      e.row_pos = m->row_pos;
      e.row_slot = m->row_slot;
      e.rope_cos = m->rope_cos;
      e.rope_sin = m->rope_sin;
      e.q_out = m->qrot;
      e.kpool = m->kpool + l * layer_elems;
      e.vpool = m->vpool + l * layer_elems;
      e.l2_next = Ly.wo;
      e.l2_next_bytes = q_o;
      CUDA_TRY(profiled(m, 0, wb_qkv, st, [&] { return launch_gemm_epi(kEpiQKV, &Ly.tm_qkv, tmx_xn, BM, e, st); }));
    }
    ap.layer_row0 = l * c.num_pages * Hkv * kPage;
    CUDA_TRY(profiled(m, 5, kv_bytes, st, [&] { return launch_attention(&m->tm_k, &m->tm_v, ap, st); }));
    {
      EpiParams e = base;
      e.N = d;
      e.K = m->q_dim;
      e.rscale = Ly.rs_o;
      e.splits = splits_for(e.N, e.K);
      e.ssq_in = nullptr;
      e.resid = m->resid;
      e.g_next = Ly.ffn_norm;
      e.xn = m->xn;
      e.ssq_out = m->ssq_b;
      e.d = d;
      e.l2_next = reinterpret_cast<const char*>(Ly.wgu) + pf_gu;
      e.l2_next_bytes = (unsigned long long)std::max(0.0, std::min(proj_pf, wb_gu - (double)pf_gu)) & ~15ull;
      CUDA_TRY(profiled(m, 1, wb_o, st, [&] { return launch_gemm_epi(kEpiResid, &Ly.tm_o, tmx_attn, BM, e, st); }));
    }
    {
      EpiParams e = base;
      e.N = 2 * F;
      e.K = d;
      e.rscale = Ly.rs_gu;
      e.splits = splits_for(e.N, e.K);
      e.ssq_in = m->ssq_b;
      e.act = m->act;
      e.ffn = F;
      e.l2_next = Ly.wdown;
      e.l2_next_bytes = (unsigned long long)std::min(proj_pf, wb_dn) & ~15ull;
      CUDA_TRY(profiled(m, 2, wb_gu, st, [&] { return launch_gemm_epi(kEpiSwiGLU, &Ly.tm_gu, tmx_xn, BM, e, st); }));
    }
    {
      EpiParams e = base;
      e.N = d;
      e.K = F;
      e.rscale = Ly.rs_down;
      e.splits = splits_for(e.N, e.K);
      e.ssq_in = nullptr;
      e.resid = m->resid;
      e.g_next = l + 1 < c.n_layers ? m->layers[l + 1].attn_norm : m->final_norm;
      e.xn = m->xn;
      e.ssq_out = m->ssq_a;
      e.d = d;
      if (l + 1 < c.n_layers) {
        e.l2_next = m->layers[l + 1].wqkv;
        e.l2_next_bytes = (unsigned long long)std::min(proj_pf, wb_qkv) & ~15ull;
      } else if (want_logits) {
        e.l2_next = m->lm_head;
        e.l2_next_bytes = (unsigned long long)std::min(proj_pf, 2.0 * c.vocab * d) & ~15ull;
      }
      CUDA_TRY(profiled(m, 3, wb_dn, st, [&] { return launch_gemm_epi(kEpiResid, &Ly.tm_down, tmx_act, BM, e, st); }));
    }
  }
  if (want_logits) {
    EpiParams e = base;
    e.N = c.vocab;
    e.K = d;
    e.rscale = m->rs_lm;
    e.splits = 1;
    e.ssq_in = m->ssq_a;
    e.logits = m->logits;
    e.inv_temp = inv_temp;
    e.tstat_max = m->tstat_max;
    e.tstat_sum = sampled ? m->tstat_sum : nullptr;
    e.tstat_arg = m->tstat_arg;
    e.tstat_stride = m->M_max;
    CUDA_TRY(profiled(m, 4, 2.0 * c.vocab * d, st, [&] { return launch_gemm_epi(kEpiLogits, &m->tm_lm, tmx_xn, BM, e, st); }));
    m->last_rows = M;
  }
  return SPEC_OK;
}

RoundAcceptParams round_params(spec_model* m, int B, int gamma, const int32_t* seq_ids, const int32_t* tok,
                               const float* q, const float* u, float inv_temp, int32_t* accepted,
                               int32_t* committed, int32_t* bonus) {
  RoundAcceptParams r{};
  r.B = B;
  r.gamma = gamma;
  r.seq_wlen = m->seq_wlen;
  r.seq_rowoff = m->seq_rowoff;
  r.cap = nullptr;
  r.V = m->cfg.vocab;
  r.inv_temp = inv_temp;
  r.logits = m->logits;
  r.n_tiles = m->cfg.vocab / 128;
  r.tstat_max = m->tstat_max;
  r.tstat_sum = m->tstat_sum;
  r.tstat_arg = m->tstat_arg;
  r.tstat_stride = m->M_max;
  r.probs = nullptr;
  r.q = q;
  r.tok = tok;
  r.x = nullptr;
  r.u = u;
  r.accepted = accepted;
  r.committed = committed;
  r.bonus = bonus;
  r.seq_ids = seq_ids;
  r.seq_ok = m->seq_ok;
  r.seq_len = m->seq_len;
  r.seq_npages = m->seq_npages;
  r.page_table = m->page_table;
  r.free_bits = m->free_bits;
  r.max_pages = m->max_pages;
  r.max_batch = m->cfg.max_batch;
  r.status = m->status;
  r.sel = nullptr;
  r.sel_max = nullptr;
  r.sel_z = nullptr;
  return r;
}

// Top-k / top-p of a sampled round: one selection launch over every window row,
// whose kept sets and softmax statistics the acceptance then uses.
spec_status adjust_round(spec_model* m, int B, int Wmax, const int32_t* top_k, const float* top_p,
                         RoundAcceptParams& rp, cudaStream_t st) {
  if (!top_k && !top_p) return SPEC_OK;
  if (m->cfg.vocab > select_max_vocab())
    return fail(SPEC_ERR_INVALID_ARG, "top-k / top-p supports vocabularies up to %d", select_max_vocab());
  SelectParams sp{};
  sp.V = m->cfg.vocab;
  sp.top_k = top_k;
  sp.top_p = top_p;
  sp.logits = m->logits;
  sp.tstat_max = m->tstat_max;
  sp.tstat_sum = m->tstat_sum;
  sp.n_tiles = m->cfg.vocab / 128;
  sp.tstat_stride = m->M_max;
  sp.inv_temp = rp.inv_temp;
  sp.seq_wlen = m->seq_wlen;
  sp.seq_rowoff = m->seq_rowoff;
  sp.sel = m->sel;
  sp.row_max = m->sel_max;
  sp.row_z = m->sel_z;
  sp.status = m->status;
  CUDA_TRY(launch_select(sp, PSource::kLogits, Wmax, B, st));
  rp.sel = m->sel;
  rp.sel_max = m->sel_max;
  rp.sel_z = m->sel_z;
  return SPEC_OK;
}

constexpr int kProfMax = 1024;

// Run `launch` bracketed by a pair of events when profiling is on.
template <typename F>
cudaError_t profiled(spec_model* m, int cls, double bytes, cudaStream_t st, F&& launch) {
  if (!m->profiling || (int)m->prof_rec.size() >= kProfMax) return launch();
  const int i = (int)m->prof_rec.size();
  cudaError_t e = cudaEventRecord(m->prof_ev[2 * i], st);
  if (e != cudaSuccess) return e;
  e = launch();
  if (e != cudaSuccess) return e;
  e = cudaEventRecord(m->prof_ev[2 * i + 1], st);
  m->prof_rec.push_back({cls, bytes});
  return e;
}

void chain_masks(int W, int* depth, uint32_t* anc) {
  for (int j = 0; j < W; ++j) {
    depth[j] = j;
    anc[j] = (j == 31) ? 0xffffffffu : ((1u << (j + 1)) - 1u);
  }
}

spec_status tree_masks(int N, const int32_t* parent, int* depth, uint32_t* anc) {
  if (!parent) return fail(SPEC_ERR_INVALID_ARG, "parent is NULL");
  if (parent[0] != -1) return fail(SPEC_ERR_INVALID_ARG, "parent[0] must be -1");
  depth[0] = 0;
  anc[0] = 1u;
  for (int c = 1; c < N; ++c) {
    if (parent[c] < 0 || parent[c] >= c) return fail(SPEC_ERR_INVALID_ARG, "parent[%d] must be in [0, %d)", c, c);
    depth[c] = depth[parent[c]] + 1;
    anc[c] = anc[parent[c]] | (1u << c);
  }
  return SPEC_OK;
}

spec_status check_model(const spec_model* m) {
  if (!m) return fail(SPEC_ERR_INVALID_ARG, "model is NULL");
  return SPEC_OK;
}

spec_status check_batch(const spec_model* m, int B, int W) {
  if (B < 1 || B > m->cfg.max_batch) return fail(SPEC_ERR_INVALID_ARG, "B=%d outside 1..%d", B, m->cfg.max_batch);
  if (W < 1 || W > m->cfg.max_width) return fail(SPEC_ERR_INVALID_ARG, "width %d outside 1..%d", W, m->cfg.max_width);
  return SPEC_OK;
}

void bump_bounds(spec_model* m, int W) {
  for (auto& v : m->host_len_bound) v = std::min<long long>(v + W, m->cfg.max_seq_len);
}

}  // namespace

// =============================================================================== C ABI
extern "C" {

const char* spec_last_error(void) { return g_err.c_str(); }

int32_t spec_max_pages_per_seq(const spec_model* m) { return m ? m->max_pages : 0; }

int32_t spec_last_launch_count(const spec_model* m) { return m ? m->last_launches : 0; }

spec_status spec_model_create(const spec_config* cfg, spec_model** out) {
  if (!cfg || !out) return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  spec_status s = validate_cfg(*cfg);
  if (s != SPEC_OK) return s;
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  CUDA_TRY(cudaGetDeviceProperties(&prop, dev));
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(SPEC_ERR_UNSUPPORTED_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                prop.major, prop.minor);
  if (!get_encode()) return fail(SPEC_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");

  auto* m = new spec_model();
  m->cfg = *cfg;
  m->device = dev;
  m->sm_count = prop.multiProcessorCount;
  const spec_config& c = m->cfg;
  m->max_pages = (c.max_seq_len + kPage - 1) / kPage;
  m->M_max = c.max_batch * c.max_width;
  m->q_dim = c.n_heads * c.head_dim;
  m->kv_dim = c.n_kv_heads * c.head_dim;
  m->qkv_n = m->q_dim + 2 * m->kv_dim;
  m->host_len_bound.assign(c.max_batch, 0);
  const int d = c.d_model, F = c.ffn_dim, V = c.vocab, hd = c.head_dim;
  const int M_max = m->M_max;

  auto bail = [&](spec_status st) {
    spec_model_destroy(m);
    return st;
  };
#define ALLOC(ptr, n)                               \
  do {                                              \
    spec_status st_ = alloc_t(m, &(ptr), (size_t)(n)); \
    if (st_ != SPEC_OK) return bail(st_);           \
  } while (0)

  ALLOC(m->embed, (size_t)V * d);
  ALLOC(m->lm_head, (size_t)V * d);
  ALLOC(m->rs_lm, V);
  ALLOC(m->final_norm, d);
  m->layers.resize(c.n_layers);
  for (auto& Ly : m->layers) {
    ALLOC(Ly.wqkv, (size_t)m->qkv_n * d);
    ALLOC(Ly.wo, (size_t)d * m->q_dim);
    ALLOC(Ly.wgu, (size_t)2 * F * d);
    ALLOC(Ly.wdown, (size_t)d * F);
    ALLOC(Ly.rs_qkv, m->qkv_n);
    ALLOC(Ly.rs_o, d);
    ALLOC(Ly.rs_gu, 2 * F);
    ALLOC(Ly.rs_down, d);
    ALLOC(Ly.attn_norm, d);
    ALLOC(Ly.ffn_norm, d);
  }
  const size_t kv_elems = (size_t)c.n_layers * c.num_pages * c.n_kv_heads * kPage * hd;
  ALLOC(m->kpool, kv_elems);
  ALLOC(m->vpool, kv_elems);
  ALLOC(m->seq_len, c.max_batch);
  ALLOC(m->seq_npages, c.max_batch);
  ALLOC(m->page_table, (size_t)c.max_batch * m->max_pages);
  ALLOC(m->free_bits, (size_t)(c.num_pages + 31) / 32);
  ALLOC(m->status, 1);
  m->M_alloc = std::max(M_max, 256);
  ALLOC(m->resid, (size_t)M_max * d);
  ALLOC(m->xn, (size_t)m->M_alloc * d);
  ALLOC(m->qrot, (size_t)M_max * m->q_dim);
  ALLOC(m->attn_out, (size_t)m->M_alloc * m->q_dim);
  ALLOC(m->act, (size_t)m->M_alloc * F);
  ALLOC(m->ssq_a, (size_t)(d / 128) * M_max);
  ALLOC(m->ssq_b, (size_t)(d / 128) * M_max);
  ALLOC(m->logits, (size_t)M_max * V);
  ALLOC(m->tstat_max, (size_t)(V / 128) * M_max);
  ALLOC(m->tstat_sum, (size_t)(V / 128) * M_max);
  ALLOC(m->tstat_arg, (size_t)(V / 128) * M_max);
  ALLOC(m->sel, M_max);
  ALLOC(m->tree_path, M_max);
  ALLOC(m->sel_max, M_max);
  ALLOC(m->sel_z, M_max);
  ALLOC(m->row_pos, M_max);
  ALLOC(m->row_slot, M_max);
  ALLOC(m->seq_start, c.max_batch);
  ALLOC(m->seq_wlen, c.max_batch);
  ALLOC(m->seq_rowoff, c.max_batch);
  ALLOC(m->seq_ok, c.max_batch);
  ALLOC(m->seq_order, c.max_batch);
  ALLOC(m->rope_cos, (size_t)c.max_seq_len * (hd / 2));
  ALLOC(m->rope_sin, (size_t)c.max_seq_len * (hd / 2));
  ALLOC(m->scratch_ids, c.max_batch);
  ALLOC(m->scratch_ids2, c.max_batch);
  ALLOC(m->scratch_lens, c.max_batch);
  ALLOC(m->scratch_tok, M_max);
  ALLOC(m->scratch_acc, c.max_batch);
  ALLOC(m->scratch_bonus, c.max_batch);
#undef ALLOC

  // RoPE angle tables: pos * theta^(-2i/hd), in double, rounded to fp32
  {
    const int half = hd / 2;
    std::vector<float> cs((size_t)c.max_seq_len * half), sn((size_t)c.max_seq_len * half);
    for (int pos = 0; pos < c.max_seq_len; ++pos)
      for (int i = 0; i < half; ++i) {
        const double a = (double)pos * std::pow((double)c.rope_theta, -2.0 * i / hd);
        cs[(size_t)pos * half + i] = (float)std::cos(a);
        sn[(size_t)pos * half + i] = (float)std::sin(a);
      }
    cudaError_t e1 = cudaMemcpy(m->rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice);
    cudaError_t e2 = cudaMemcpy(m->rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice);
    if (e1 != cudaSuccess || e2 != cudaSuccess) return bail(fail(SPEC_ERR_CUDA, "rope table upload failed"));
  }
  // gains default to 1
  {
    std::vector<float> ones(d, 1.f);
    cudaMemcpy(m->final_norm, ones.data(), d * 4, cudaMemcpyHostToDevice);
    for (auto& Ly : m->layers) {
      cudaMemcpy(Ly.attn_norm, ones.data(), d * 4, cudaMemcpyHostToDevice);
      cudaMemcpy(Ly.ffn_norm, ones.data(), d * 4, cudaMemcpyHostToDevice);
    }
  }
  // tensor maps
  bool ok = true;
  for (auto& Ly : m->layers) {
    ok &= make_map(&Ly.tm_qkv, Ly.wqkv, d, m->qkv_n, 64, 128);
    ok &= make_map(&Ly.tm_o, Ly.wo, m->q_dim, d, 64, 128);
    ok &= make_map(&Ly.tm_gu, Ly.wgu, d, 2 * F, 64, 128);
    ok &= make_map(&Ly.tm_down, Ly.wdown, F, d, 64, 128);
  }
  ok &= make_map(&m->tm_lm, m->lm_head, d, V, 64, 128);
  for (int i = 0; i < kNumBM; ++i) {
    ok &= make_map(&m->tm_xn[i], m->xn, d, m->M_alloc, 64, kBMs[i]);
    ok &= make_map(&m->tm_attn[i], m->attn_out, m->q_dim, m->M_alloc, 64, kBMs[i]);
    ok &= make_map(&m->tm_act[i], m->act, F, m->M_alloc, 64, kBMs[i]);
  }
  const uint64_t kv_rows = (uint64_t)c.n_layers * c.num_pages * c.n_kv_heads * kPage;
  for (int i = 0; i < kPairBoxes; ++i) {
    ok &= make_map(&m->tm_xn2[i], m->xn, d, m->M_alloc, 64, 8 * (i + 1));
    ok &= make_map(&m->tm_attn2[i], m->attn_out, m->q_dim, m->M_alloc, 64, 8 * (i + 1));
    ok &= make_map(&m->tm_act2[i], m->act, F, m->M_alloc, 64, 8 * (i + 1));
  }
  m->pair_ok = m->qkv_n % 256 == 0 && d % 256 == 0 && (2 * F) % 256 == 0 && V % 256 == 0;
  ok &= make_map(&m->tm_k, m->kpool, hd, kv_rows, 64, 64);
  ok &= make_map(&m->tm_v, m->vpool, hd, kv_rows, 64, 64);
  if (!ok) return bail(fail(SPEC_ERR_CUDA, "tensor map encoding failed"));

  cudaError_t e = launch_init_state(m->seq_len, m->seq_npages, m->page_table, m->free_bits, c.max_batch,
                                    m->max_pages, c.num_pages, nullptr);
  if (e != cudaSuccess) return bail(fail(SPEC_ERR_CUDA, "state init failed: %s", cudaGetErrorString(e)));
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return bail(fail(SPEC_ERR_CUDA, "create sync failed: %s", cudaGetErrorString(e)));
  *out = m;
  return SPEC_OK;
}

void spec_model_destroy(spec_model* m) {
  if (!m) return;
  cudaDeviceSynchronize();
  for (auto e : m->prof_ev) cudaEventDestroy(e);
  for (void* p : m->allocs) cudaFree(p);
  delete m;
}

spec_status spec_model_set_weight(spec_model* m, spec_weight which, int32_t layer, const void* src, int64_t n_elems,
                                  void* stream) {
  if (spec_status s = check_model(m)) return s;
  if (!src) return fail(SPEC_ERR_INVALID_ARG, "src is NULL");
  const spec_config& c = m->cfg;
  const int d = c.d_model, F = c.ffn_dim;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool per_layer = which >= SPEC_W_ATTN_NORM;
  if (per_layer && (layer < 0 || layer >= c.n_layers)) return fail(SPEC_ERR_INVALID_ARG, "layer %d out of range", layer);
  auto expect = [&](long long n) -> spec_status {
    if (n_elems != n) return fail(SPEC_ERR_INVALID_ARG, "weight %d: got %lld elements, expected %lld", (int)which,
                                  (long long)n_elems, n);
    return SPEC_OK;
  };
  auto copy = [&](void* dst, size_t bytes) -> spec_status {
    CUDA_TRY(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, st));
    return SPEC_OK;
  };
  spec_model::Layer* Ly = per_layer ? &m->layers[layer] : nullptr;
  // matrices: copy the bf16 rows into place, then re-encode them in place as fp16 x 2^e
  auto encode = [&](void* base, int K, int n_rows, int block, int block_stride, int row0,
                    float* rscale) -> spec_status {
    CUDA_TRY(launch_encode_rows(static_cast<uint16_t*>(base), K, n_rows, block, block_stride, row0, rscale, st));
    return SPEC_OK;
  };
  switch (which) {
    case SPEC_W_EMBED:
      if (auto s = expect((long long)c.vocab * d)) return s;
      return copy(m->embed, (size_t)n_elems * 2);
    case SPEC_W_LM_HEAD:
      if (auto s = expect((long long)c.vocab * d)) return s;
      if (auto s = copy(m->lm_head, (size_t)n_elems * 2)) return s;
      return encode(m->lm_head, d, c.vocab, c.vocab, 0, 0, m->rs_lm);
    case SPEC_W_FINAL_NORM:
      if (auto s = expect(d)) return s;
      return copy(m->final_norm, (size_t)d * 4);
    case SPEC_W_ATTN_NORM:
      if (auto s = expect(d)) return s;
      return copy(Ly->attn_norm, (size_t)d * 4);
    case SPEC_W_FFN_NORM:
      if (auto s = expect(d)) return s;
      return copy(Ly->ffn_norm, (size_t)d * 4);
    case SPEC_W_WQ:
      if (auto s = expect((long long)m->q_dim * d)) return s;
      if (auto s = copy(Ly->wqkv, (size_t)n_elems * 2)) return s;
      return encode(Ly->wqkv, d, m->q_dim, m->q_dim, 0, 0, Ly->rs_qkv);
    case SPEC_W_WK:
      if (auto s = expect((long long)m->kv_dim * d)) return s;
      if (auto s = copy(Ly->wqkv + (size_t)m->q_dim * d, (size_t)n_elems * 2)) return s;
      return encode(Ly->wqkv, d, m->kv_dim, m->kv_dim, 0, m->q_dim, Ly->rs_qkv);
    case SPEC_W_WV:
      if (auto s = expect((long long)m->kv_dim * d)) return s;
      if (auto s = copy(Ly->wqkv + (size_t)(m->q_dim + m->kv_dim) * d, (size_t)n_elems * 2)) return s;
      return encode(Ly->wqkv, d, m->kv_dim, m->kv_dim, 0, m->q_dim + m->kv_dim, Ly->rs_qkv);
    case SPEC_W_WO:
      if (auto s = expect((long long)d * m->q_dim)) return s;
      if (auto s = copy(Ly->wo, (size_t)n_elems * 2)) return s;
      return encode(Ly->wo, m->q_dim, d, d, 0, 0, Ly->rs_o);
    case SPEC_W_DOWN:
      if (auto s = expect((long long)d * F)) return s;
      if (auto s = copy(Ly->wdown, (size_t)n_elems * 2)) return s;
      return encode(Ly->wdown, F, d, d, 0, 0, Ly->rs_down);
    case SPEC_W_GATE:
    case SPEC_W_UP: {
      if (auto s = expect((long long)F * d)) return s;
      // 64-row blocks interleaved: block j of gate -> rows 128j..128j+63, of up -> 128j+64..128j+127
      const size_t blk = (size_t)64 * d * 2;
      const int off = which == SPEC_W_UP ? 64 : 0;
      char* dst = reinterpret_cast<char*>(Ly->wgu) + (which == SPEC_W_UP ? blk : 0);
      CUDA_TRY(cudaMemcpy2DAsync(dst, 2 * blk, src, blk, blk, F / 64, cudaMemcpyDefault, st));
      return encode(Ly->wgu, d, F, 64, 128, off, Ly->rs_gu);
    }
    default:
      return fail(SPEC_ERR_INVALID_ARG, "unknown weight kind %d", (int)which);
  }
}

spec_status spec_seq_reset(spec_model* m, int32_t n, const int32_t* seq_ids_host, void* stream) {
  if (spec_status s = check_model(m)) return s;
  if (n < 1 || n > m->cfg.max_batch || !seq_ids_host) return fail(SPEC_ERR_INVALID_ARG, "bad reset list");
  for (int i = 0; i < n; ++i) {
    if (seq_ids_host[i] < 0 || seq_ids_host[i] >= m->cfg.max_batch)
      return fail(SPEC_ERR_INVALID_ARG, "sequence id %d out of range", seq_ids_host[i]);
    m->host_len_bound[seq_ids_host[i]] = 0;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaMemcpyAsync(m->scratch_ids, seq_ids_host, n * 4, cudaMemcpyHostToDevice, st));
  ResetParams rp{m->scratch_ids, n, m->seq_len, m->seq_npages, m->page_table, m->free_bits, m->max_pages};
  CUDA_TRY(launch_seq_reset(rp, st));
  CUDA_TRY(cudaStreamSynchronize(st));  // the host id list may be reused by the caller
  return SPEC_OK;
}

spec_status spec_prefill(spec_model* m, int32_t B, const int32_t* seq_ids, const int32_t* tokens, int32_t stride,
                         const int32_t* lens_host, void* stream) {
  if (spec_status s = check_model(m)) return s;
  if (B < 1 || B > m->cfg.max_batch) return fail(SPEC_ERR_INVALID_ARG, "B out of range");
  if (!seq_ids || !tokens || !lens_host) return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
  int max_len = 0;
  for (int b = 0; b < B; ++b) {
    if (lens_host[b] < 1 || lens_host[b] > stride) return fail(SPEC_ERR_INVALID_ARG, "lens[%d] = %d", b, lens_host[b]);
    if (lens_host[b] - 1 > m->cfg.max_seq_len) return fail(SPEC_ERR_CAPACITY, "prompt longer than max_seq_len");
    max_len = std::max(max_len, (int)lens_host[b]);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int W = m->cfg.max_width;
  // sequences sorted by cached length, longest first: the active set of every full
  // window is then a prefix of this order
  std::vector<int32_t> perm(B), add(B);
  for (int b = 0; b < B; ++b) {
    perm[b] = b;
    add[b] = lens_host[b] - 1;
  }
  std::stable_sort(perm.begin(), perm.end(), [&](int a, int b) { return lens_host[a] > lens_host[b]; });
  // Reserve every prompt's pages first, in the caller's sequence order.
  CUDA_TRY(cudaMemcpyAsync(m->scratch_acc, add.data(), B * 4, cudaMemcpyHostToDevice, st));
  CUDA_TRY(launch_alloc_to_len(seq_ids, m->scratch_acc, B, 1, m->seq_len, m->seq_npages, m->page_table, m->free_bits,
                               m->max_pages, m->cfg.num_pages, m->cfg.max_batch, m->status, st));
  CUDA_TRY(cudaMemcpyAsync(m->scratch_lens, perm.data(), B * 4, cudaMemcpyHostToDevice, st));
  CUDA_TRY(cudaStreamSynchronize(st));  // perm and add are host buffers
  int depth[16];
  uint32_t anc[16];
  g_launch_count = 0;
  for (int c0 = 0;; c0 += W) {
    int k = 0;
    while (k < B && lens_host[perm[k]] - 1 >= c0 + W) ++k;
    if (k == 0) break;
    chain_masks(W, depth, anc);
    CUDA_TRY(launch_gather_tokens(tokens, stride, m->scratch_lens, k, c0, W, m->scratch_tok, seq_ids, m->scratch_ids2,
                                  st));
    if (auto s = forward(m, k, W, m->scratch_ids2, m->scratch_tok, depth, anc, false, false, 1.f, st)) return s;
    CUDA_TRY(launch_commit_all(m->scratch_ids2, m->seq_ok, k, W, m->cfg.max_batch, m->seq_len, st));
  }
  for (int i = 0; i < B; ++i) {  // the ragged tail of each prompt
    const int n_cache = lens_host[perm[i]] - 1;
    const int r = n_cache % W;
    if (r == 0) continue;
    const int c0 = n_cache - r;
    chain_masks(r, depth, anc);
    CUDA_TRY(launch_gather_tokens(tokens, stride, m->scratch_lens + i, 1, c0, r, m->scratch_tok, seq_ids,
                                  m->scratch_ids2, st));
    if (auto s = forward(m, 1, r, m->scratch_ids2, m->scratch_tok, depth, anc, false, false, 1.f, st)) return s;
    CUDA_TRY(launch_commit_all(m->scratch_ids2, m->seq_ok, 1, r, m->cfg.max_batch, m->seq_len, st));
  }
  m->last_launches = g_launch_count;
  // host bound: sequences ids are on the device; raise every slot's bound
  for (auto& v : m->host_len_bound) v = std::min<long long>(std::max<long long>(v, 0) + max_len, m->cfg.max_seq_len);
  return SPEC_OK;
}

// Shared set-up of the tree acceptance parameters.
TreeParams tree_params(spec_model* m, int B, int n_nodes, const int32_t* seq_ids, const int32_t* tok,
                       const int32_t* parent_host, int32_t* accepted, int32_t* committed, int32_t* bonus) {
  TreeParams tp{};
  tp.B = B;
  tp.N = n_nodes;
  tp.V = m->cfg.vocab;
  for (int j = 0; j < 16; ++j) tp.parent[j] = j < n_nodes ? parent_host[j] : -1;
  tp.tok = tok;
  tp.accepted = accepted;
  tp.committed = committed;
  tp.bonus = bonus;
  tp.seq_ids = seq_ids;
  tp.seq_ok = m->seq_ok;
  tp.seq_len = m->seq_len;
  tp.seq_npages = m->seq_npages;
  tp.page_table = m->page_table;
  tp.free_bits = m->free_bits;
  tp.max_pages = m->max_pages;
  tp.max_batch = m->cfg.max_batch;
  tp.kpool = m->kpool;
  tp.vpool = m->vpool;
  tp.n_layers = m->cfg.n_layers;
  tp.num_pages = m->cfg.num_pages;
  tp.Hkv = m->cfg.n_kv_heads;
  tp.hd = m->cfg.head_dim;
  tp.status = m->status;
  return tp;
}

spec_status spec_verify_tree_sampled(spec_model* m, int32_t B, int32_t n_nodes, const int32_t* seq_ids,
                                     const int32_t* tok, const int32_t* parent_host, const float* q, const float* u,
                                     float temperature, const int32_t* top_k, const float* top_p, int32_t* accepted,
                                     int32_t* committed, int32_t* bonus, void* stream) {
  if (spec_status s = check_model(m)) return s;
  if (spec_status s = check_batch(m, B, n_nodes)) return s;
  if (!seq_ids || !tok || !u || !accepted || !committed || !bonus) return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
  if (!(temperature > 0.f) || std::isinf(temperature))
    return fail(SPEC_ERR_INVALID_ARG, "sampled tree verify needs temperature > 0");
  int depth[16];
  uint32_t anc[16];
  if (auto s = tree_masks(n_nodes, parent_host, depth, anc)) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  g_launch_count = 0;
  const float inv_t = 1.f / temperature;
  if (auto s = forward(m, B, n_nodes, seq_ids, tok, depth, anc, true, true, inv_t, st)) return s;
  TreeParams tp = tree_params(m, B, n_nodes, seq_ids, tok, parent_host, accepted, committed, bonus);
  tp.stats = round_params(m, B, n_nodes - 1, seq_ids, tok, nullptr, u, inv_t, accepted, committed, bonus);
  if (auto s = adjust_round(m, B, n_nodes, top_k, top_p, tp.stats, st)) return s;
  tp.q = q;
  tp.u = u;
  tp.path = m->tree_path;
  CUDA_TRY(launch_accept_tree_sampled(tp, st));
  bump_bounds(m, n_nodes);
  m->last_launches = g_launch_count;
  return SPEC_OK;
}

spec_status spec_score(spec_model* m, int32_t B, int32_t W, const int32_t* seq_ids, const int32_t* tok,
                       const int32_t* parent_host, float* logits_out, void* stream) {
  if (spec_status s = check_model(m)) return s;
  if (spec_status s = check_batch(m, B, W)) return s;
  if (!seq_ids || !tok) return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
  int depth[16];
  uint32_t anc[16];
  if (parent_host) {
    if (auto s = tree_masks(W, parent_host, depth, anc)) return s;
  } else {
    chain_masks(W, depth, anc);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  g_launch_count = 0;
  if (auto s = forward(m, B, W, seq_ids, tok, depth, anc, true, false, 1.f, st)) return s;
  if (logits_out)
    CUDA_TRY(cudaMemcpyAsync(logits_out, m->logits, (size_t)B * W * m->cfg.vocab * 4, cudaMemcpyDeviceToDevice, st));
  m->last_launches = g_launch_count;
  return SPEC_OK;
}

spec_status spec_decode_step(spec_model* m, int32_t B, const int32_t* seq_ids, const int32_t* tok, float temperature,
                             const int32_t* top_k, const float* top_p, const float* u, int32_t* next_tok,
                             void* stream) {
  if (spec_status s = check_model(m)) return s;
  if (spec_status s = check_batch(m, B, 1)) return s;
  if (!seq_ids || !tok || !next_tok) return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
  if (!(temperature >= 0.f) || std::isinf(temperature)) return fail(SPEC_ERR_INVALID_ARG, "bad temperature");
  const bool sampled = temperature > 0.f;
  if (sampled && !u) return fail(SPEC_ERR_INVALID_ARG, "sampled decode needs u (no greedy fallback)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int depth[16];
  uint32_t anc[16];
  chain_masks(1, depth, anc);
  g_launch_count = 0;
  const float inv_t = sampled ? 1.f / temperature : 1.f;
  if (auto s = forward(m, B, 1, seq_ids, tok, depth, anc, true, sampled, inv_t, st)) return s;
  RoundAcceptParams rp = round_params(m, B, 0, seq_ids, tok, nullptr, u, inv_t, m->scratch_acc, next_tok,
                                      m->scratch_bonus);
  if (sampled)
    if (auto s = adjust_round(m, B, 1, top_k, top_p, rp, st)) return s;
  CUDA_TRY(launch_accept_round(rp, sampled, st));
  bump_bounds(m, 1);
  m->last_launches = g_launch_count;
  return SPEC_OK;
}

spec_status spec_verify_step(spec_model* m, int32_t B, int32_t gamma, const int32_t* seq_ids, const int32_t* tok,
                             const float* q, const float* u, float temperature, const int32_t* top_k,
                             const float* top_p, int32_t* accepted, int32_t* committed, int32_t* bonus,
                             void* stream) {
  if (spec_status s = check_model(m)) return s;
  if (gamma < 0) return fail(SPEC_ERR_INVALID_ARG, "gamma < 0");
  const int W = gamma + 1;
  if (spec_status s = check_batch(m, B, W)) return s;
  if (!seq_ids || !tok || !accepted || !committed || !bonus) return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
  if (!(temperature >= 0.f) || std::isinf(temperature)) return fail(SPEC_ERR_INVALID_ARG, "bad temperature");
  const bool sampled = temperature > 0.f;
  if (sampled && (!u || (gamma > 0 && !q)))
    return fail(SPEC_ERR_INVALID_ARG, "sampled verify needs q and u (no greedy fallback)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int depth[16];
  uint32_t anc[16];
  chain_masks(W, depth, anc);
  g_launch_count = 0;
  const float inv_t = sampled ? 1.f / temperature : 1.f;
  if (auto s = forward(m, B, W, seq_ids, tok, depth, anc, true, sampled, inv_t, st)) return s;
  RoundAcceptParams rp = round_params(m, B, gamma, seq_ids, tok, q, u, inv_t, accepted, committed, bonus);
  if (sampled)
    if (auto s = adjust_round(m, B, W, top_k, top_p, rp, st)) return s;
  CUDA_TRY(launch_accept_round(rp, sampled, st));
  bump_bounds(m, W);
  m->last_launches = g_launch_count;
  return SPEC_OK;
}

spec_status spec_verify_ragged(spec_model* m, int32_t B, int32_t gamma, const int32_t* seq_ids, const int32_t* tok,
                               const int32_t* verify_lens, int32_t total_rows, int32_t mode, const float* q,
                               const float* u, float temperature, const int32_t* top_k, const float* top_p,
                               int32_t* accepted, int32_t* committed, int32_t* bonus, void* stream) {
  if (spec_status s = check_model(m)) return s;
  if (gamma < 0) return fail(SPEC_ERR_INVALID_ARG, "gamma < 0");
  const int W = gamma + 1;
  if (spec_status s = check_batch(m, B, W)) return s;
  if (!seq_ids || !tok || !verify_lens || !accepted || !committed || !bonus)
    return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
  if (mode != SPEC_RAGGED_CAP_ACCEPT && mode != SPEC_RAGGED_COMPACT) return fail(SPEC_ERR_INVALID_ARG, "bad mode");
  if (mode == SPEC_RAGGED_COMPACT && (total_rows < B || total_rows > B * W))
    return fail(SPEC_ERR_INVALID_ARG, "total_rows %d outside [B, B*(gamma+1)]", total_rows);
  if (!(temperature >= 0.f) || std::isinf(temperature)) return fail(SPEC_ERR_INVALID_ARG, "bad temperature");
  const bool sampled = temperature > 0.f;
  if (sampled && (!u || (gamma > 0 && !q)))
    return fail(SPEC_ERR_INVALID_ARG, "sampled verify needs q and u (no greedy fallback)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int depth[16];
  uint32_t anc[16];
  chain_masks(W, depth, anc);
  g_launch_count = 0;
  const float inv_t = sampled ? 1.f / temperature : 1.f;
  if (mode == SPEC_RAGGED_COMPACT) {
    if (auto s = forward(m, B, W, seq_ids, tok, depth, anc, true, sampled, inv_t, st, verify_lens, total_rows))
      return s;
  } else {
    if (auto s = forward(m, B, W, seq_ids, tok, depth, anc, true, sampled, inv_t, st)) return s;
  }
  RoundAcceptParams rp = round_params(m, B, gamma, seq_ids, tok, q, u, inv_t, accepted, committed, bonus);
  if (mode == SPEC_RAGGED_CAP_ACCEPT) rp.cap = verify_lens;
  if (sampled)
    if (auto s = adjust_round(m, B, W, top_k, top_p, rp, st)) return s;
  CUDA_TRY(launch_accept_round(rp, sampled, st));
  bump_bounds(m, W);
  m->last_launches = g_launch_count;
  return SPEC_OK;
}

spec_status spec_verify_tree_step(spec_model* m, int32_t B, int32_t n_nodes, const int32_t* seq_ids,
                                  const int32_t* tok, const int32_t* parent_host, int32_t* accepted,
                                  int32_t* committed, int32_t* bonus, void* stream) {
  if (spec_status s = check_model(m)) return s;
  if (spec_status s = check_batch(m, B, n_nodes)) return s;
  if (!seq_ids || !tok || !accepted || !committed || !bonus) return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
  int depth[16];
  uint32_t anc[16];
  if (auto s = tree_masks(n_nodes, parent_host, depth, anc)) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  g_launch_count = 0;
  if (auto s = forward(m, B, n_nodes, seq_ids, tok, depth, anc, true, false, 1.f, st)) return s;
  TreeParams tp = tree_params(m, B, n_nodes, seq_ids, tok, parent_host, accepted, committed, bonus);
  tp.stats = round_params(m, B, n_nodes - 1, seq_ids, tok, nullptr, nullptr, 1.f, accepted, committed, bonus);
  CUDA_TRY(launch_accept_tree(tp, st));
  bump_bounds(m, n_nodes);
  m->last_launches = g_launch_count;
  return SPEC_OK;
}

spec_status spec_accept_probs(int32_t B, int32_t gamma, int32_t V, const float* p, const float* q, const int32_t* x,
                              const float* u, int32_t* accepted, int32_t* committed, int32_t* bonus, void* stream) {
  if (B < 1 || gamma < 0 || gamma + 1 > kMaxWidth || V < 1) return fail(SPEC_ERR_INVALID_ARG, "bad shape");
  if (!p || !u || (gamma > 0 && (!q || !x)) || !accepted || !committed || !bonus)
    return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
  // the model round's acceptance kernel, reading the given probabilities
  RoundAcceptParams rp{};
  rp.B = B;
  rp.gamma = gamma;
  rp.V = V;
  rp.inv_temp = 1.f;
  rp.probs = p;
  rp.q = q;
  rp.x = x;
  rp.u = u;
  rp.accepted = accepted;
  rp.committed = committed;
  rp.bonus = bonus;
  CUDA_TRY(launch_accept_round_probs(rp, static_cast<cudaStream_t>(stream)));
  return SPEC_OK;
}

spec_status spec_adjust_probs(int32_t rows, int32_t V, const float* p, float* p_out, const int32_t* top_k,
                              const float* top_p, int32_t rows_per_setting, void* stream) {
  if (rows < 1 || V < 1 || rows_per_setting < 1) return fail(SPEC_ERR_INVALID_ARG, "bad shape");
  if (rows > 65535) return fail(SPEC_ERR_INVALID_ARG, "at most 65535 rows per call");
  if (V > select_max_vocab())
    return fail(SPEC_ERR_INVALID_ARG, "top-k / top-p supports vocabularies up to %d", select_max_vocab());
  if (!p || !p_out) return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
  SelectParams sp{};
  sp.V = V;
  sp.top_k = top_k;
  sp.top_p = top_p;
  sp.p_in = p;
  sp.p_out = p_out;
  sp.rows_per_set = rows_per_setting;
  sp.status = nullptr;
  CUDA_TRY(launch_select(sp, PSource::kProbs, rows, 1, static_cast<cudaStream_t>(stream)));
  return SPEC_OK;
}

spec_status spec_accept_tree_probs(int32_t B, int32_t n_nodes, int32_t V, const float* p, const float* q,
                                  const int32_t* tok, const int32_t* parent_host, const float* u, int32_t* accepted,
                                  int32_t* committed, int32_t* bonus, void* stream) {
  if (B < 1 || n_nodes < 1 || n_nodes > kMaxWidth || V < 1) return fail(SPEC_ERR_INVALID_ARG, "bad shape");
  if (!p || !tok || !parent_host || !u || !accepted || !committed || !bonus)
    return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
  int depth[16];
  uint32_t anc[16];
  if (auto s = tree_masks(n_nodes, parent_host, depth, anc)) return s;
  TreeParams tp{};
  tp.B = B;
  tp.N = n_nodes;
  tp.V = V;
  for (int j = 0; j < 16; ++j) tp.parent[j] = j < n_nodes ? parent_host[j] : -1;
  tp.tok = tok;
  tp.accepted = accepted;
  tp.committed = committed;
  tp.bonus = bonus;
  tp.q = q;
  tp.u = u;
  tp.probs = p;
  CUDA_TRY(launch_accept_tree_sampled(tp, static_cast<cudaStream_t>(stream)));
  return SPEC_OK;
}

spec_status spec_accept_greedy(int32_t B, int32_t gamma, int32_t V, const float* logits, const int32_t* x,
                               int32_t* accepted, int32_t* committed, int32_t* bonus, void* stream) {
  if (B < 1 || gamma < 0 || gamma + 1 > kMaxWidth || V < 1) return fail(SPEC_ERR_INVALID_ARG, "bad shape");
  if (!logits || (gamma > 0 && !x) || !accepted || !committed || !bonus)
    return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
  AcceptParams ap{};
  ap.B = B;
  ap.gamma = gamma;
  ap.V = V;
  ap.rows = logits;
  ap.tok = x;
  ap.row_argmax = nullptr;  // argmax taken inside the accept kernel
  ap.accepted = accepted;
  ap.committed = committed;
  ap.bonus = bonus;
  CUDA_TRY(launch_accept_greedy(ap, static_cast<cudaStream_t>(stream)));
  return SPEC_OK;
}

spec_status spec_get_kv_state(spec_model* m, int32_t n, const int32_t* seq_ids_host, int32_t* seq_len_host,
                              int32_t* page_table_host) {
  if (spec_status s = check_model(m)) return s;
  if (n < 1 || !seq_ids_host || !seq_len_host || !page_table_host) return fail(SPEC_ERR_INVALID_ARG, "bad arguments");
  CUDA_TRY(cudaDeviceSynchronize());
  for (int i = 0; i < n; ++i) {
    const int s = seq_ids_host[i];
    if (s < 0 || s >= m->cfg.max_batch) return fail(SPEC_ERR_INVALID_ARG, "sequence id out of range");
    CUDA_TRY(cudaMemcpy(&seq_len_host[i], m->seq_len + s, 4, cudaMemcpyDeviceToHost));
    CUDA_TRY(cudaMemcpy(page_table_host + (size_t)i * m->max_pages, m->page_table + (size_t)s * m->max_pages,
                        (size_t)m->max_pages * 4, cudaMemcpyDeviceToHost));
  }
  return SPEC_OK;
}

spec_status spec_read_kv(spec_model* m, int32_t layer, int32_t seq_id, int32_t t0, int32_t n, uint16_t* k_host,
                         uint16_t* v_host) {
  if (spec_status s = check_model(m)) return s;
  const spec_config& c = m->cfg;
  if (layer < 0 || layer >= c.n_layers || seq_id < 0 || seq_id >= c.max_batch || t0 < 0 || n < 0 ||
      t0 + n > m->max_pages * kPage || !k_host || !v_host)
    return fail(SPEC_ERR_INVALID_ARG, "bad arguments");
  CUDA_TRY(cudaDeviceSynchronize());
  std::vector<int32_t> pt(m->max_pages);
  CUDA_TRY(cudaMemcpy(pt.data(), m->page_table + (size_t)seq_id * m->max_pages, m->max_pages * 4,
                      cudaMemcpyDeviceToHost));
  const int hd = c.head_dim, Hkv = c.n_kv_heads;
  for (int t = t0; t < t0 + n; ++t) {
    const int pg = pt[t / kPage];
    if (pg < 0) return fail(SPEC_ERR_INVALID_ARG, "slot %d has no page", t);
    for (int h = 0; h < Hkv; ++h) {
      const size_t off = ((((size_t)layer * c.num_pages + pg) * Hkv + h) * kPage + t % kPage) * hd;
      const size_t dst = ((size_t)(t - t0) * Hkv + h) * hd;
      CUDA_TRY(cudaMemcpy(k_host + dst, m->kpool + off, hd * 2, cudaMemcpyDeviceToHost));
      CUDA_TRY(cudaMemcpy(v_host + dst, m->vpool + off, hd * 2, cudaMemcpyDeviceToHost));
    }
  }
  return SPEC_OK;
}

spec_status spec_debug_logits(spec_model* m, float* out, int64_t max_elems, void* stream) {
  if (spec_status s = check_model(m)) return s;
  const long long n = (long long)m->last_rows * m->cfg.vocab;
  if (!out || max_elems < n) return fail(SPEC_ERR_INVALID_ARG, "output too small (%lld needed)", n);
  CUDA_TRY(cudaMemcpyAsync(out, m->logits, (size_t)n * 4, cudaMemcpyDefault, static_cast<cudaStream_t>(stream)));
  return SPEC_OK;
}

spec_status spec_debug_wait_probe(spec_model* m, int64_t budget_cycles, void* stream) {
  if (spec_status s = check_model(m)) return s;
  if (budget_cycles < 1 || budget_cycles > 4000000000ll) return fail(SPEC_ERR_INVALID_ARG, "budget out of range");
  CUDA_TRY(launch_wait_probe(m->status, (unsigned long long)budget_cycles, static_cast<cudaStream_t>(stream)));
  return SPEC_OK;
}

spec_status spec_kv_fill_random(spec_model* m, int32_t n, const int32_t* seq_ids_host, const int32_t* lens_host,
                                uint64_t seed, float scale, void* stream) {
  if (spec_status s = check_model(m)) return s;
  if (n < 1 || n > m->cfg.max_batch || !seq_ids_host || !lens_host) return fail(SPEC_ERR_INVALID_ARG, "bad arguments");
  for (int i = 0; i < n; ++i) {
    if (seq_ids_host[i] < 0 || seq_ids_host[i] >= m->cfg.max_batch) return fail(SPEC_ERR_INVALID_ARG, "bad id");
    if (lens_host[i] < 0 || lens_host[i] > m->cfg.max_seq_len) return fail(SPEC_ERR_CAPACITY, "length too long");
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaMemcpyAsync(m->scratch_ids, seq_ids_host, n * 4, cudaMemcpyHostToDevice, st));
  CUDA_TRY(cudaMemcpyAsync(m->scratch_lens, lens_host, n * 4, cudaMemcpyHostToDevice, st));
  ResetParams rp{m->scratch_ids, n, m->seq_len, m->seq_npages, m->page_table, m->free_bits, m->max_pages};
  CUDA_TRY(launch_seq_reset(rp, st));
  CUDA_TRY(launch_alloc_to_len(m->scratch_ids, m->scratch_lens, n, 0, m->seq_len, m->seq_npages, m->page_table,
                               m->free_bits, m->max_pages, m->cfg.num_pages, m->cfg.max_batch, m->status, st));
  CUDA_TRY(launch_kv_fill_pages(m->kpool, m->vpool, m->page_table, m->seq_npages, m->max_pages, m->scratch_ids, n,
                                m->cfg.n_layers, m->cfg.num_pages, m->cfg.n_kv_heads, m->cfg.head_dim, seed, scale,
                                st));
  CUDA_TRY(cudaStreamSynchronize(st));
  for (int i = 0; i < n; ++i) m->host_len_bound[seq_ids_host[i]] = lens_host[i];
  return SPEC_OK;
}

spec_status spec_kv_write(spec_model* m, int32_t seq_id, int32_t n_tokens, const uint16_t* k, const uint16_t* v,
                          void* stream) {
  if (spec_status s = check_model(m)) return s;
  const spec_config& c = m->cfg;
  if (seq_id < 0 || seq_id >= c.max_batch) return fail(SPEC_ERR_INVALID_ARG, "sequence id %d out of range", seq_id);
  if (n_tokens < 0 || n_tokens > c.max_seq_len) return fail(SPEC_ERR_CAPACITY, "n_tokens %d outside 0..max_seq_len", n_tokens);
  if (n_tokens > 0 && (!k || !v)) return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15u)
    return fail(SPEC_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t ids[1] = {seq_id}, lens[1] = {n_tokens};
  CUDA_TRY(cudaMemcpyAsync(m->scratch_ids, ids, 4, cudaMemcpyHostToDevice, st));
  CUDA_TRY(cudaMemcpyAsync(m->scratch_lens, lens, 4, cudaMemcpyHostToDevice, st));
  ResetParams rp{m->scratch_ids, 1, m->seq_len, m->seq_npages, m->page_table, m->free_bits, m->max_pages};
  CUDA_TRY(launch_seq_reset(rp, st));
  CUDA_TRY(launch_alloc_to_len(m->scratch_ids, m->scratch_lens, 1, 0, m->seq_len, m->seq_npages, m->page_table,
                               m->free_bits, m->max_pages, c.num_pages, c.max_batch, m->status, st));
  CUDA_TRY(launch_kv_write(m->kpool, m->vpool, m->page_table, m->max_pages, seq_id, n_tokens,
                           reinterpret_cast<const act_t*>(k), reinterpret_cast<const act_t*>(v), c.n_layers,
                           c.num_pages, c.n_kv_heads, c.head_dim, st));
  CUDA_TRY(cudaStreamSynchronize(st));  // ids and lens are host buffers
  m->host_len_bound[seq_id] = n_tokens;
  return SPEC_OK;
}

spec_status spec_set_profiling(spec_model* m, int32_t enable) {
  if (spec_status s = check_model(m)) return s;
  if (enable && m->prof_ev.empty()) {
    m->prof_ev.resize(2 * kProfMax);
    for (auto& e : m->prof_ev) CUDA_TRY(cudaEventCreate(&e));
  }
  m->profiling = enable != 0;
  m->prof_rec.clear();
  return SPEC_OK;
}

spec_status spec_read_profile(spec_model* m, double* ms, int64_t* launches, double* bytes) {
  if (spec_status s = check_model(m)) return s;
  if (!ms || !launches || !bytes) return fail(SPEC_ERR_INVALID_ARG, "NULL argument");
  CUDA_TRY(cudaDeviceSynchronize());
  for (size_t i = 0; i < m->prof_rec.size(); ++i) {
    float t = 0.f;
    CUDA_TRY(cudaEventElapsedTime(&t, m->prof_ev[2 * i], m->prof_ev[2 * i + 1]));
    const int c = m->prof_rec[i].cls;
    ms[c] += t;
    launches[c] += 1;
    bytes[c] += m->prof_rec[i].bytes;
  }
  m->prof_rec.clear();
  return SPEC_OK;
}

spec_status spec_sync_status(spec_model* m, void* stream) {
  if (spec_status s = check_model(m)) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaStreamSynchronize(st));
  CUDA_TRY(cudaGetLastError());
  int code = 0;
  CUDA_TRY(cudaMemcpy(&code, m->status, 4, cudaMemcpyDeviceToHost));
  CUDA_TRY(cudaMemset(m->status, 0, 4));
  // The host's per-sequence length bounds (launch shapes only: attention split,
  // key groups, L2 prefetch budget) grow by the window on every call; the stream
  // is idle here, so take the exact lengths instead.
  std::vector<int32_t> lens(m->cfg.max_batch);
  CUDA_TRY(cudaMemcpy(lens.data(), m->seq_len, lens.size() * 4, cudaMemcpyDeviceToHost));
  for (size_t i = 0; i < lens.size(); ++i) m->host_len_bound[i] = std::max(0, (int)lens[i]);
  // The only device-side SPEC_ERR_UNSUPPORTED: a CTA pair of the pair projection
  // kernel not placed on the two SMs of one TPC (it computed nothing).  Later
  // calls use the single-CTA tensor-core tiles instead.
  if (code == SPEC_ERR_UNSUPPORTED) m->pair_ok = false;
  if (code != 0) return fail((spec_status)code, "device reported status %d", code);
  return SPEC_OK;
}

}  // extern "C"
