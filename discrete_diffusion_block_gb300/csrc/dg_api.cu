// C ABI of the decoder library (declared in include/dg.h): model state, the
// paged KV cache, the per-layer launch sequence and the canvas loop.
//
// Procedure (DiffusionGemma report §1-§4 and §3.4; blog "Once Written, a
// Prefix Becomes History"): the prompt is encoded once with causal attention
// and its K/V cached; each canvas of C tokens starts as uniform random ids
// and is refined by denoising forwards in which the canvas sees the whole
// cached prefix and itself bidirectionally; the sampler commits confident or
// stable positions and re-noises the rest until the canvas is finished; one
// extra forward then encodes the finished canvas and appends its K/V, after
// which it is read-only prefix.
//
// KV layout: per layer, K and V pools [n_pages][Hkv][page_size][hd] bf16 with
// a page table mapping logical page j (tokens j*page_size ...) to a physical
// page.  During denoising the canvas K/V of the current layer are written
// into the slots the canvas will occupy once committed (positions
// prefix .. prefix + C - 1): attention then treats prefix and canvas keys
// uniformly, and the KV-append forward overwrites those slots with the
// clean canvas's K/V.
#include <chrono>
#include <cstdarg>
#include <map>
#include <mutex>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "internal.h"

using dg::bf16;

namespace {

thread_local std::string g_err;

int fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

#define CK(call)                                                                          \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess) {                                                              \
      cudaGetLastError(); /* a failed launch must not be reported again by a later call */ \
      return fail(DG_ECUDA, "%s failed: %s", #call, cudaGetErrorString(e_));              \
    }                                                                                     \
  } while (0)

#define CKR(call)                                                                         \
  do {                                                                                    \
    int r_ = (call);                                                                      \
    if (r_ != DG_OK) return r_;                                                           \
  } while (0)

constexpr int kPrefillChunk = 2048;

struct Layer {
  bf16 *wqkv = nullptr, *wo = nullptr, *wr = nullptr, *wgu = nullptr, *wd = nullptr;
  uint8_t *wgu8 = nullptr;  // expert_fp8: W_gate / W_up as e4m3 operand tiles
  int *kw = nullptr;        // expert_fp8: their rows' scale exponents [E][2][F]
  float *attn_norm = nullptr, *moe_norm = nullptr;
};

double now_s() {
  return std::chrono::duration<double>(std::chrono::steady_clock::now().time_since_epoch()).count();
}

}  // namespace

struct dg_model {
  dg_config cfg;
  dg_sampler_config sc;
  bool borrowed_weights = false;  // weights are the caller's (dg_init_model's weights[])
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  std::vector<void *> allocs;
  // weights
  bf16 *embed = nullptr, *lm_head = nullptr;
  float *final_norm = nullptr;
  std::vector<Layer> layers;
  // KV cache
  bf16 *k_pool = nullptr, *v_pool = nullptr;
  int n_pages = 0;
  size_t layer_pool_elems = 0;
  int *page_table = nullptr;
  std::vector<int> page_table_host;
  float *cos_t = nullptr, *sin_t = nullptr;
  // scratch for up to Tmax tokens
  int Tmax = 0;
  int *ids = nullptr;
  float *h = nullptr;
  bf16 *xq = nullptr;  // the attention-norm output, as operand tiles (the QKV operand)
  bf16 *xn = nullptr, *xn_lo = nullptr, *q = nullptr, *o = nullptr, *act = nullptr,
       *x_tiles = nullptr;  // act and x_tiles: expert-FFN operand tiles per work item
  unsigned long long *moe_stats = nullptr;  // device: experts touched, rows routed
  int *route_bar = nullptr;                  // device, kGridBarInts: grid barrier of the fused routing + scatter
  float *ffn_part = nullptr;                 // device: partial-sum slots of split gate/up units
  int *kx = nullptr;                         // expert_fp8: scale exponents of the expert input rows
  int moe_input_rows = 0, moe_input_layer = -1;  // the rows xn holds: the last MoE input
  float *gates = nullptr;
  bf16 *y = nullptr;  // [T*k][d]: expert outputs per sorted pair row
  float *xchg = nullptr;  // split-K partial exchange of the projection GEMMs
  int *topk = nullptr, *offs = nullptr, *gcount = nullptr, *slot_row = nullptr, *work = nullptr,
      *n_work = nullptr;
  int max_work = 0;
  std::vector<int> routing_rows;  // rows routed by the last forward, per layer
  void *attn_ws = nullptr;
  size_t attn_ws_bytes = 0;
  void *partials = nullptr;
  // canvas state
  int *x = nullptr, *last = nullptr, *stable = nullptr, *argmax = nullptr, *gumbel = nullptr,
      *done_dev = nullptr;
  uint8_t *committed = nullptr;
  float *conf = nullptr;
  int *done_host = nullptr;  // pinned, 2 ints (done, error word)
  int prompt_len = 0, prefix_len = 0, canvas_index = 0, step = 0;
  // Lockstep batching: B requests, each with n_pages_req KV pages (request b
  // owns physical pages b * n_pages_req ...), its own prompt and prefix, and
  // its canvas at rows [b C, b C + C) of every per-position array.  With
  // B = 1 the request's lengths are also prompt_len / prefix_len above.
  int B = 1, n_pages_req = 0;
  std::vector<int> prompt_lens, prefix_lens;
  int *req_done = nullptr, *req_nk = nullptr, *batch_counter = nullptr;  // device, BatchCtl
  bool prefilled = false, canvas_active = false, canvas_done = false;
  // profiling: launch counts always, event-timed device ms when prof_on
  bool prof_on = false;
  double prof_ms[DG_K_CLASSES] = {};
  int64_t prof_launches[DG_K_CLASSES] = {};
  struct ProfRec {
    int cls;
    cudaEvent_t a, b;
  };
  std::vector<ProfRec> prof_pending;
  std::vector<cudaEvent_t> prof_free;
  // CUDA graphs of the denoising step, one per (prefix length, profiling on)
  struct StepGraph {
    cudaGraphExec_t exec = nullptr;
    std::vector<ProfRec> recs;  // event pairs captured as graph nodes
    int64_t launches[DG_K_CLASSES] = {};
  };
  std::map<std::pair<int, int>, StepGraph> graphs;
  StepGraph *capturing = nullptr;
  // Device-side canvas loops, one per prefix length: a graph whose WHILE
  // node repeats the captured step until the sampler reports the canvas done.
  struct LoopGraph {
    cudaGraphExec_t exec = nullptr;
    int64_t launches[DG_K_CLASSES] = {};  // kernels of one iteration
  };
  std::map<int, LoopGraph> loop_graphs;
  dg::LoopCtl loop_ctl{};  // set while a loop body is being captured
  int64_t host_syncs = 0;  // device -> host synchronisations of the canvas loops
  bool eager_step_done = false;  // the first step runs eagerly (sets kernel attributes)
  dg::StepParams *dyn_dev = nullptr, *dyn_host = nullptr;  // per-step sampler words

  int alloc_count = 0;    // device allocations made by this model
  // Host-side fault injection (DG_FAULT, read at dg_init_model; nothing is
  // done to the GPU): allocation n (1-based) fails with DG_ENOMEM, kernel
  // launch n fails with DG_ECUDA before it is made, or every KV capacity
  // check reports a full pool (DG_ECAPACITY).
  int fail_alloc_at = 0;
  int launch_count = 0, fail_launch_at = 0;
  bool fault_kvfull = false;
  template <class T>
  int alloc(T **p, size_t n) {
    void *v = nullptr;
    if (n == 0) n = 1;
    if (++alloc_count == fail_alloc_at)
      return fail(DG_ENOMEM, "device allocation %d failed (injected by DG_FAULT)", alloc_count);
    if (cudaMalloc(&v, n * sizeof(T)) != cudaSuccess) {
      cudaGetLastError();
      return fail(DG_ENOMEM, "cudaMalloc of %zu bytes failed", n * sizeof(T));
    }
    allocs.push_back(v);
    *p = (T *)v;
    return DG_OK;
  }
  bf16 *kpool(int L) { return k_pool + (size_t)L * layer_pool_elems; }
  bf16 *vpool(int L) { return v_pool + (size_t)L * layer_pool_elems; }
};

namespace {

cudaEvent_t prof_event(dg_model *m) {
  if (!m->prof_free.empty()) {
    cudaEvent_t e = m->prof_free.back();
    m->prof_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return e;
}

// Events of a step being captured belong to its graph (they are replayed with
// it); other events come from the model's reuse pool.
cudaEvent_t prof_new_event(dg_model *m) {
  if (!m->capturing) return prof_event(m);
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return e;
}

// Inside a capture a plain record only orders the capture; the external
// flag turns it into an event-record node that timestamps each replay.
void prof_record(dg_model *m, cudaEvent_t e) {
  if (m->capturing)
    cudaEventRecordWithFlags(e, m->stream, cudaEventRecordExternal);
  else
    cudaEventRecord(e, m->stream);
}

cudaEvent_t prof_begin(dg_model *m) {
  if (!m->prof_on) return nullptr;
  cudaEvent_t a = prof_new_event(m);
  if (a) prof_record(m, a);
  return a;
}

void prof_end(dg_model *m, int cls, int n_kernels, cudaEvent_t a) {
  (m->capturing ? m->capturing->launches : m->prof_launches)[cls] += n_kernels;
  if (!a) return;
  cudaEvent_t b = prof_new_event(m);
  if (!b) {
    if (m->capturing) cudaEventDestroy(a); else m->prof_free.push_back(a);
    return;
  }
  prof_record(m, b);
  (m->capturing ? m->capturing->recs : m->prof_pending).push_back({cls, a, b});
}

// After a replay has finished: add the graph's launches and event times.
void prof_collect_graph(dg_model *m, const dg_model::StepGraph &g) {
  for (int i = 0; i < DG_K_CLASSES; ++i) m->prof_launches[i] += g.launches[i];
  for (const auto &r : g.recs) {
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) m->prof_ms[r.cls] += ms;
    cudaGetLastError();
  }
}

void destroy_graphs(dg_model *m) {
  for (auto &kv : m->loop_graphs)
    if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
  m->loop_graphs.clear();
  for (auto &kv : m->graphs) {
    if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
    for (auto &r : kv.second.recs) {
      cudaEventDestroy(r.a);
      cudaEventDestroy(r.b);
    }
  }
  m->graphs.clear();
}

// Fold finished event pairs into the per-class totals (stream already synced).
void prof_collect(dg_model *m) {
  for (auto &r : m->prof_pending) {
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) m->prof_ms[r.cls] += ms;
    cudaGetLastError();
    m->prof_free.push_back(r.a);
    m->prof_free.push_back(r.b);
  }
  m->prof_pending.clear();
}

// Launch `call` (one or more kernels of class `cls`) with profiling brackets.
#define KL(cls, nk, call)                                                                 \
  do {                                                                                    \
    if (m->fail_launch_at && ++m->launch_count == m->fail_launch_at)                      \
      return fail(DG_ECUDA, "launch %d failed (injected by DG_FAULT=badcall)", m->launch_count); \
    cudaEvent_t a_ = prof_begin(m);                                                       \
    cudaError_t e_ = (call);                                                              \
    prof_end(m, (cls), (nk), a_);                                                         \
    if (e_ != cudaSuccess) {                                                              \
      cudaGetLastError();                                                                 \
      return fail(DG_ECUDA, "%s failed: %s", #call, cudaGetErrorString(e_));              \
    }                                                                                     \
  } while (0)

#define SYNC(m)                                                                           \
  do {                                                                                    \
    CK(cudaStreamSynchronize((m)->stream));                                               \
    prof_collect(m);                                                                      \
  } while (0)

int validate(const dg_config *c, const dg_sampler_config *s) {
  if (!c || !s) return fail(DG_EINVAL, "null config");
  if (c->n_layers < 1 || c->d_model < 64 || c->d_model % 64)
    return fail(DG_EINVAL, "d_model must be a positive multiple of 64");
  if (c->head_dim != 64 && c->head_dim != 128) return fail(DG_EINVAL, "head_dim must be 64 or 128");
  if (c->n_kv_heads < 1 || c->n_q_heads % c->n_kv_heads)
    return fail(DG_EINVAL, "n_q_heads must be a multiple of n_kv_heads");
  if ((c->n_q_heads * c->head_dim) % 64)
    return fail(DG_EINVAL, "n_q_heads*head_dim must be a multiple of 64");
  if (c->n_experts < 1 || c->n_experts > 256) return fail(DG_EINVAL, "n_experts must be in [1, 256]");
  if (c->top_k < 1 || c->top_k > 16 || c->top_k > c->n_experts)
    return fail(DG_EINVAL, "top_k must be in [1, min(16, n_experts)]");
  if (c->d_ff < 64 || c->d_ff % 64) return fail(DG_EINVAL, "d_ff must be a positive multiple of 64");
  if (c->vocab < 256 || c->vocab % 256) return fail(DG_EINVAL, "vocab must be a positive multiple of 256");
  if (c->page_size < 64 || c->page_size % 64)
    return fail(DG_EINVAL, "page_size must be a positive multiple of 64");
  if (c->max_requests < 0 || c->max_requests > dg::kMaxRequests)
    return fail(DG_EINVAL, "max_requests must be in [0, %d]", dg::kMaxRequests);
  if (c->expert_fp8 != 0 && c->expert_fp8 != 1) return fail(DG_EINVAL, "expert_fp8 must be 0 or 1");
  if (c->expert_fp8 && c->d_model % 128) return fail(DG_EINVAL, "expert_fp8 needs d_model a multiple of 128");
  if (s->canvas_len < 1 || s->canvas_len > 1024) return fail(DG_EINVAL, "canvas_len must be in [1, 1024]");
  if (c->max_context < s->canvas_len) return fail(DG_EINVAL, "max_context smaller than one canvas");
  if (s->budget_N < 1 || s->budget_N > 65535) return fail(DG_EINVAL, "budget_N must be in [1, 65535]");
  if (s->stable_steps < 1) return fail(DG_EINVAL, "stable_steps must be >= 1");
  if (!(s->temp_start > 0.0f) || !(s->temp_end > 0.0f))
    return fail(DG_EINVAL, "temp_start and temp_end must be > 0");
  return DG_OK;
}

// All layers over T tokens already embedded in m->h, at the positions of
// `rows` (one request's tokens from pos0[0], or n_req requests' rows, see
// dg::RowSet); K/V go to the cache at those positions through page table
// `ptab` (the request's slice, or the whole table with rows.n_req > 1).
// kv_only_last: the last layer only needs its K/V (KV-append and prefill).
int run_layers(dg_model *m, int T, const dg::RowSet &rows, const int *ptab, int causal, bool kv_only_last) {
  const dg_config &c = m->cfg;
  const int d = c.d_model, qd = c.n_q_heads * c.head_dim;
  cudaStream_t st = m->stream;
  const bool fuse_norm = d <= 4096;  // the MoE combine also writes the next layer's input norm
  for (int L = 0; L < c.n_layers; ++L) {
    const Layer &W = m->layers[L];
    if (L == 0 || !fuse_norm)
      KL(DG_K_RMSNORM, 1, dg::rmsnorm_rows(m->xq, m->h, W.attn_norm, T, d, c.rms_eps, st, nullptr, true));
    dg::QkvOut qo{m->q, m->kpool(L), m->vpool(L), ptab, rows, c.page_size,
                  c.n_q_heads, c.n_kv_heads, c.head_dim, m->cos_t, m->sin_t};
    int *err = m->done_dev + 1;
    KL(DG_K_QKV_ROPE, 1, dg::gemm_qkv(m->xq, W.wqkv, T, d, qo, err, m->xchg, st));
    if (kv_only_last && L == c.n_layers - 1) break;
    dg::AttnShape as{rows.pos0[0], rows.n_req > 1 ? rows.rows_per_req : T, c.n_q_heads, c.n_kv_heads,
                     c.head_dim, c.page_size, causal, m->n_pages};
    as.n_req = rows.n_req;
    as.pages_per_req = rows.pages_per_req;
    for (int b = 0; b < rows.n_req; ++b) as.req_prefix[b] = rows.pos0[b];
    KL(DG_K_ATTENTION, dg::attention_launch_count(as),
       dg::attention(m->q, m->kpool(L), m->vpool(L), ptab, as, m->o, m->attn_ws,
                     m->attn_ws_bytes, st, err, true));
    KL(DG_K_O_PROJ, 1, dg::gemm_residual(m->o, W.wo, T, qd, d, m->h, err, m->xchg, st));
    int *topk = m->topk + (size_t)L * m->Tmax * c.top_k;
    m->routing_rows[L] = T;
    m->moe_input_rows = T;
    m->moe_input_layer = L;
    int nl = 0;  // routing and scatter: one launch, or two when the routing grid exceeds the machine
    const dg::Fp8Experts fx{W.wgu8, W.kw, m->kx};
    KL(DG_K_ROUTE, nl,
       dg::moe_route_scatter(m->h, W.moe_norm, c.rms_eps, m->xn, W.wr, T, d, c.n_experts, c.top_k, topk,
                             m->gates, m->slot_row, m->gcount, m->x_tiles, m->offs, m->work, m->n_work,
                             m->max_work, m->route_bar, err, st, m->moe_stats, &nl,
                             c.expert_fp8 ? &fx : nullptr));
    const int rows = T * c.top_k;
    KL(DG_K_EXPERT_FFN, 1,
       dg::moe_ffn(m->x_tiles, rows, W.wgu, W.wd, m->offs, m->work, m->n_work, m->max_work,
                   c.n_experts, d, c.d_ff, m->act, m->y, err, st, c.expert_fp8 ? &fx : nullptr, m->ffn_part,
                   (int)dg::moe_ffn_part_slots()));
    if (fuse_norm && L + 1 < c.n_layers) {
      KL(DG_K_COMBINE, 1,
         dg::moe_combine_norm(m->h, m->y, m->gates, m->slot_row, T, c.top_k, d, m->layers[L + 1].attn_norm,
                              c.rms_eps, m->xq, st));
    } else {
      KL(DG_K_COMBINE, 1, dg::moe_combine(m->h, m->y, m->gates, m->slot_row, T, c.top_k, d, true, st));
    }
  }
  return DG_OK;
}

int fill_model_weights(dg_model *m) {
  const dg_config &c = m->cfg;
  const int d = c.d_model, qd = c.n_q_heads * c.head_dim, kd = c.n_kv_heads * c.head_dim;
  const uint64_t s = c.weight_seed;
  const float sd = c.init_std;
  cudaStream_t st = m->stream;
  CK(dg::fill_weights(m->embed, (uint64_t)c.vocab * d, s, 1, 0, sd, st));
  CK(dg::fill_tiled_weights(m->lm_head, c.vocab, d, c.vocab, c.vocab, 2, 2, 2, s, sd, st));
  CK(dg::fill_const(m->final_norm, d, 1.0f, st));
  for (int L = 0; L < c.n_layers; ++L) {
    const uint32_t b = 100u + 16u * (uint32_t)L;
    Layer &W = m->layers[L];
    CK(dg::fill_tiled_weights(W.wqkv, qd + 2 * kd, d, qd, qd + kd, b + 0, b + 1, b + 2, s, sd, st));
    CK(dg::fill_tiled_weights(W.wo, d, qd, d, d, b + 3, b + 3, b + 3, s, sd, st));
    CK(dg::fill_moe_weights(W.wr, W.wgu, W.wd, d, c.n_experts, c.d_ff, L, s, sd, st));
    CK(dg::fill_const(W.attn_norm, d, 1.0f, st));
    CK(dg::fill_const(W.moe_norm, d, 1.0f, st));
  }
  return DG_OK;
}

int alloc_model(dg_model *m, const void *const *weights) {
  const dg_config &c = m->cfg;
  const int d = c.d_model, qd = c.n_q_heads * c.head_dim, kd = c.n_kv_heads * c.head_dim;
  const int E = c.n_experts, F = c.d_ff, k = c.top_k, C = m->sc.canvas_len;
  m->layers.resize(c.n_layers);
  if (weights) {
    const int n = 3 + 7 * c.n_layers;
    for (int i = 0; i < n; ++i)
      if (!weights[i] || ((uintptr_t)weights[i] & 15))
        return fail(DG_EINVAL, "borrowed weight %d is null or not 16-byte aligned", i);
    m->embed = (bf16 *)weights[DG_W_EMBED];
    m->lm_head = (bf16 *)weights[DG_W_LM_HEAD];
    m->final_norm = (float *)weights[DG_W_FINAL_NORM];
    for (int L = 0; L < c.n_layers; ++L) {
      const void *const *w = weights + 3 + 7 * L;
      Layer &W = m->layers[L];
      W.wqkv = (bf16 *)w[DG_W_WQKV - 3];
      W.wo = (bf16 *)w[DG_W_WO - 3];
      W.wr = (bf16 *)w[DG_W_ROUTER - 3];
      W.wgu = (bf16 *)w[DG_W_GATE_UP - 3];
      W.wd = (bf16 *)w[DG_W_DOWN - 3];
      W.attn_norm = (float *)w[DG_W_ATTN_NORM - 3];
      W.moe_norm = (float *)w[DG_W_MOE_NORM - 3];
    }
    m->borrowed_weights = true;
  } else {
    CKR(m->alloc(&m->embed, (size_t)c.vocab * d));
    CKR(m->alloc(&m->lm_head, (size_t)c.vocab * d));
    CKR(m->alloc(&m->final_norm, d));
    for (auto &W : m->layers) {
      CKR(m->alloc(&W.wqkv, (size_t)(qd + 2 * kd) * d));
      CKR(m->alloc(&W.wo, (size_t)d * qd));
      CKR(m->alloc(&W.wr, (size_t)E * d));
      CKR(m->alloc(&W.wgu, (size_t)E * 2 * F * d));
      CKR(m->alloc(&W.wd, (size_t)E * d * F));
      CKR(m->alloc(&W.attn_norm, d));
      CKR(m->alloc(&W.moe_norm, d));
    }
  }
  m->n_pages_req = dg::ceil_div(c.max_context, c.page_size);
  m->n_pages = m->B * m->n_pages_req;
  m->layer_pool_elems = (size_t)m->n_pages * kd * c.page_size;
  CKR(m->alloc(&m->k_pool, m->layer_pool_elems * c.n_layers));
  CKR(m->alloc(&m->v_pool, m->layer_pool_elems * c.n_layers));
  // cache slots never written yet are read (and weighted by zero) at the tail
  // of a key tile: they must hold finite values
  CK(cudaMemset(m->k_pool, 0, m->layer_pool_elems * c.n_layers * sizeof(bf16)));
  CK(cudaMemset(m->v_pool, 0, m->layer_pool_elems * c.n_layers * sizeof(bf16)));
  CKR(m->alloc(&m->page_table, m->n_pages));
  m->page_table_host.resize(m->n_pages);
  for (int i = 0; i < m->n_pages; ++i) m->page_table_host[i] = i;  // request b: its own range, in order
  CKR(m->alloc(&m->cos_t, (size_t)c.max_context * c.head_dim / 2));
  CKR(m->alloc(&m->sin_t, (size_t)c.max_context * c.head_dim / 2));

  const int BC = m->B * C;  // rows of a batched canvas forward
  const int T = m->Tmax = BC > kPrefillChunk ? BC : kPrefillChunk;
  CKR(m->alloc(&m->ids, T));
  CKR(m->alloc(&m->h, (size_t)T * d));
  CKR(m->alloc(&m->xn, (size_t)T * d));
  CKR(m->alloc(&m->xq, (size_t)T * d));
  CKR(m->alloc(&m->xn_lo, (size_t)BC * d));
  CKR(m->alloc(&m->moe_stats, 2));
  CKR(m->alloc(&m->ffn_part, dg::moe_ffn_part_slots() * (dg::kFfnPartSlotBytes / 4)));
  CKR(m->alloc(&m->route_bar, dg::kGridBarInts));
  CK(cudaMemset(m->route_bar, 0, dg::kGridBarInts * sizeof(int)));
  CKR(m->alloc(&m->q, (size_t)T * qd));
  CKR(m->alloc(&m->o, (size_t)T * qd));
  CKR(m->alloc(&m->xchg, dg::gemm_xchg_bytes() / sizeof(float)));
  CKR(m->alloc(&m->topk, (size_t)c.n_layers * T * k));  // per-layer routing record
  m->routing_rows.assign(c.n_layers, 0);
  CKR(m->alloc(&m->gates, (size_t)T * k));
  m->max_work = (int)dg::moe_max_work(T, k, E, dg::kExpertTileRows);
  CKR(m->alloc(&m->offs, E + 1));
  CKR(m->alloc(&m->gcount, dg::moe_group_count_ints(T, E)));
  CKR(m->alloc(&m->slot_row, (size_t)T * k));
  if (c.expert_fp8) CKR(m->alloc(&m->kx, (size_t)T * k));
  CKR(m->alloc(&m->work, dg::moe_work_ints(T, k, E, dg::kExpertTileRows)));
  CKR(m->alloc(&m->n_work, 1));
  CKR(m->alloc(&m->act, dg::moe_item_tile_elems(m->max_work, F)));
  CKR(m->alloc(&m->x_tiles, dg::moe_item_tile_elems(m->max_work, d)));
  CKR(m->alloc(&m->y, (size_t)T * k * d));
  size_t ws = 0;
  const int shapes[3][2] = {{c.max_context - C, C}, {0, C},
                            {c.max_context - T > 0 ? c.max_context - T : 0, T}};
  for (auto &sh : shapes) {
    dg::AttnShape as{sh[0], sh[1], c.n_q_heads, c.n_kv_heads, c.head_dim, c.page_size, 0};
    const size_t b = dg::attention_workspace_bytes(as);
    if (b > ws) ws = b;
  }
  m->attn_ws_bytes = ws;
  CKR(m->alloc((unsigned char **)&m->attn_ws, ws));
  CKR(m->alloc((unsigned char **)&m->partials, (size_t)BC * (c.vocab / dg::kVocabTile) * 20));
  CKR(m->alloc(&m->x, BC));
  CKR(m->alloc(&m->last, BC));
  CKR(m->alloc(&m->stable, BC));
  CKR(m->alloc(&m->argmax, BC));
  CKR(m->alloc(&m->gumbel, BC));
  CKR(m->alloc(&m->req_done, m->B));
  CKR(m->alloc(&m->req_nk, m->B));
  CKR(m->alloc(&m->batch_counter, 1));
  CK(cudaMemset(m->batch_counter, 0, sizeof(int)));
  // [0] canvas done, [1] error word of bounded device waits, [2] bad page index
  CKR(m->alloc(&m->done_dev, 3));
  CK(cudaMemset(m->done_dev, 0, 3 * sizeof(int)));
  CKR(m->alloc(&m->committed, BC));
  CKR(m->alloc(&m->conf, BC));
  if (cudaMallocHost(&m->done_host, 2 * sizeof(int)) != cudaSuccess ||
      cudaMallocHost(&m->dyn_host, sizeof(dg::StepParams)) != cudaSuccess) {
    cudaGetLastError();
    return fail(DG_ENOMEM, "cudaMallocHost failed");
  }
  CKR(m->alloc(&m->dyn_dev, 1));
  return DG_OK;
}

// A nonzero device error word: a bounded wait that gave up, or (codes from
// kShapeErrorBase on) a kernel that found itself launched without its
// cluster shape and returned before doing anything.
int device_fail(int code) {
  if (code >= dg::kShapeErrorBase)
    return fail(DG_ECUDA, "a kernel ran without the cluster shape it was launched with (code %d)", code);
  return fail(DG_ETIMEOUT, "a bounded device-side wait gave up (code %d)", code);
}

// expert_fp8: the e4m3 copy of every layer's W_gate / W_up and their rows'
// scale exponents, made from the bf16 weights (seeded or borrowed).
int quantize_expert_weights(dg_model *m) {
  const dg_config &c = m->cfg;
  const int E = c.n_experts, F = c.d_ff, d = c.d_model;
  for (auto &W : m->layers) {
    CKR(m->alloc(&W.wgu8, (size_t)E * 2 * F * d));
    CKR(m->alloc(&W.kw, (size_t)E * 2 * F));
    CK(dg::quantize_rows_e4m3(W.wgu, W.wgu8, W.kw, 2 * E, F, d, m->stream));
  }
  return DG_OK;
}

int check_model(dg_model *m) {
  if (!m) return fail(DG_EINVAL, "null model");
  return DG_OK;
}

// Synchronise the stream and report a bounded device-side wait that gave up
// in the work since the last check (the error word is then cleared).
int sync_check(dg_model *m) {
  CK(cudaMemcpyAsync(m->done_host, m->done_dev, 2 * sizeof(int), cudaMemcpyDeviceToHost, m->stream));
  SYNC(m);
  if (m->done_host[1]) {
    const int code = m->done_host[1];
    CK(cudaMemsetAsync(m->done_dev + 1, 0, sizeof(int), m->stream));
    SYNC(m);
    return device_fail(code);
  }
  return DG_OK;
}

// Check request b's prompt (host) against the vocabulary and its KV capacity.
int check_prompt(dg_model *m, const int32_t *prompt, int32_t n) {
  const dg_config &c = m->cfg;
  if (n < 0 || (n > 0 && !prompt)) return fail(DG_EINVAL, "bad prompt");
  if (m->fault_kvfull) return fail(DG_ECAPACITY, "KV pool full (injected by DG_FAULT=kvfull)");
  if (n + m->sc.canvas_len > c.max_context)
    return fail(DG_ECAPACITY, "prompt of %d tokens plus a canvas exceeds max_context %d", n,
                c.max_context);
  for (int i = 0; i < n; ++i)
    if (prompt[i] < 0 || prompt[i] >= c.vocab) return fail(DG_EINVAL, "prompt id %d out of range", prompt[i]);
  return DG_OK;
}

// Encode request b's prompt into its KV pages (causal), in chunks of Tmax.
// Its launches go without programmatic dependent launch even when DG_PDL=1
// asks for it: with it, encoding long prompts (chunks of 2048 tokens after a
// prefix of tens of thousands) stalled on the GB300 (one bounded wait of the
// attention gave up, and one run did not return).
int encode_prompt(dg_model *m, int b, const int32_t *prompt, int32_t n) {
  struct PdlOff {
    PdlOff() { dg::pdl_suspend(true); }
    ~PdlOff() { dg::pdl_suspend(false); }
  } pdl_off;
  const dg_config &c = m->cfg;
  const int *ptab = m->page_table + (size_t)b * m->n_pages_req;
  for (int p0 = 0; p0 < n; p0 += m->Tmax) {
    const int T = n - p0 < m->Tmax ? n - p0 : m->Tmax;
    CK(cudaMemcpyAsync(m->ids, prompt + p0, sizeof(int) * T, cudaMemcpyHostToDevice, m->stream));
    KL(DG_K_EMBED, 1, dg::embed_rows(m->h, m->embed, m->ids, T, c.d_model, m->stream));
    dg::RowSet rows;
    rows.pos0[0] = p0;
    CKR(run_layers(m, T, rows, ptab, 1, true));
    CKR(sync_check(m));  // the host prompt buffer and m->ids are reused by the next chunk
  }
  return DG_OK;
}

void reset_generation(dg_model *m) {
  m->prompt_len = m->prefix_len = m->prompt_lens[0];
  m->prefix_lens = m->prompt_lens;
  m->canvas_index = 0;
  m->prefilled = true;
  m->canvas_active = m->canvas_done = false;
}

int prefill_impl(dg_model *m, const int32_t *prompt, int32_t n) {
  CKR(check_prompt(m, prompt, n));
  CKR(encode_prompt(m, 0, prompt, n));
  m->prompt_lens.assign(1, n);
  reset_generation(m);
  return DG_OK;
}

// The rows of the current canvases: one request's canvas after its prefix,
// or (B > 1) every request's canvas after its own prefix.
dg::RowSet canvas_rows(dg_model *m) {
  dg::RowSet rows;
  rows.n_req = m->B;
  rows.rows_per_req = m->B > 1 ? m->sc.canvas_len : 0;
  rows.pages_per_req = m->B > 1 ? m->n_pages_req : 0;
  for (int b = 0; b < m->B; ++b) rows.pos0[b] = m->prefix_lens[b];
  return rows;
}

// Denoising forward of the current canvas(es) up to the final norm (in m->xn).
int canvas_forward(dg_model *m) {
  const dg_config &c = m->cfg;
  const int T = m->B * m->sc.canvas_len;
  KL(DG_K_EMBED, 1, dg::embed_rows(m->h, m->embed, m->x, T, c.d_model, m->stream));
  CKR(run_layers(m, T, canvas_rows(m), m->page_table, 0, false));
  // final norm kept to ~16 bits (hi + lo bf16), as the LM head's operand tiles
  KL(DG_K_RMSNORM, 1,
     dg::rmsnorm_rows(m->xn, m->h, m->final_norm, T, c.d_model, c.rms_eps, m->stream, m->xn_lo, true));
  m->moe_input_rows = 0;  // xn now holds the final norm
  return DG_OK;
}

// fp32(1 / tau_n) of step n under the linear annealing schedule (in double).
float annealed_inv_tau(const dg_sampler_config &s, int n) {
  double tau = s.temp_start;
  if (s.budget_N > 1) tau += ((double)s.temp_end - (double)s.temp_start) * (n - 1) / (s.budget_N - 1);
  return (float)(1.0 / tau);
}

int begin_canvas(dg_model *m) {
  if (!m->prefilled) return fail(DG_ESTATE, "dg_prefill must come first");
  if (m->canvas_done) return fail(DG_ESTATE, "canvas finished: call dg_commit_canvas");
  if (!m->canvas_active) {
    if (m->fault_kvfull) return fail(DG_ECAPACITY, "KV pool full (injected by DG_FAULT=kvfull)");
    for (int b = 0; b < m->B; ++b)
      if (m->prefix_lens[b] + m->sc.canvas_len > m->cfg.max_context)
        return fail(DG_ECAPACITY, "no room for another canvas (prefix %d, max_context %d)",
                    m->prefix_lens[b], m->cfg.max_context);
    KL(DG_K_CANVAS_INIT, 1,
       dg::canvas_init(m->x, m->committed, m->last, m->stable, m->sc.canvas_len, m->cfg.vocab,
                       m->sc.sample_seed, m->canvas_index, m->stream, m->B));
    if (m->B > 1) CK(cudaMemsetAsync(m->req_nk, 0, sizeof(int) * m->B, m->stream));
    m->step = 0;
    m->canvas_active = true;
  }
  return DG_OK;
}

// The kernels of one denoising step after canvas initialisation: forward,
// LM head with the fused vocab reduction, merge, commit rule.  Step-varying
// sampler words are read from m->dyn_dev, so the sequence can be captured.
int step_launches(dg_model *m) {
  const dg_config &c = m->cfg;
  const dg_sampler_config &s = m->sc;
  const int C = s.canvas_len, T = m->B * C;
  CKR(canvas_forward(m));
  KL(DG_K_LM_HEAD, 1,
     dg::gemm_lm_head_partials(m->xn, m->xn_lo, m->lm_head, T, c.d_model, c.vocab, s.sample_seed,
                               m->canvas_index, m->step, 1.0f, m->partials, m->done_dev + 1, m->stream,
                               m->dyn_dev, nullptr, m->B > 1 ? C : 0));
  KL(DG_K_SAMPLER_MERGE, 1,
     dg::sampler_merge(m->partials, T, c.vocab, m->argmax, m->conf, m->gumbel, m->stream));
  dg::BatchCtl bt;
  if (m->B > 1) bt = dg::BatchCtl{m->B, m->req_done, m->req_nk, m->batch_counter};
  KL(DG_K_SAMPLER_RULE, 1,
     dg::sampler_rule(m->argmax, m->conf, m->gumbel, C, m->step, s.budget_N, s.stable_steps,
                      s.adaptive, s.conf_threshold, m->x, m->committed, m->last, m->stable,
                      m->done_dev, m->stream, m->dyn_dev, m->loop_ctl, bt));
  return DG_OK;
}

// Graphs of a step are valid for one set of prefix lengths: a single
// request's prefix, or (B > 1, requests advancing together) the canvas index.
int graph_key(const dg_model *m) { return m->B > 1 ? -1 - m->canvas_index : m->prefix_len; }

// Capture step_launches() into a graph for the current prefix length.
int capture_step(dg_model *m, dg_model::StepGraph *g) {
  CK(cudaStreamBeginCapture(m->stream, cudaStreamCaptureModeThreadLocal));
  m->capturing = g;
  const int r = step_launches(m);
  m->capturing = nullptr;
  cudaGraph_t graph = nullptr;
  const cudaError_t e = cudaStreamEndCapture(m->stream, &graph);
  if (r != DG_OK) {
    if (graph) cudaGraphDestroy(graph);
    return r;
  }
  if (e != cudaSuccess) return fail(DG_ECUDA, "graph capture failed: %s", cudaGetErrorString(e));
  const cudaError_t ei = cudaGraphInstantiate(&g->exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ei != cudaSuccess) return fail(DG_ECUDA, "graph instantiation failed: %s", cudaGetErrorString(ei));
  return DG_OK;
}

// The step words of step n of the current canvas to the device.
int put_step_params(dg_model *m, int n) {
  const dg_sampler_config &s = m->sc;
  m->dyn_host->ctr2 = dg::gumbel_ctr2(m->canvas_index, n);
  m->dyn_host->key0 = (uint32_t)s.sample_seed;
  m->dyn_host->key1 = (uint32_t)(s.sample_seed >> 32);
  m->dyn_host->step = n;
  m->dyn_host->inv_tau = annealed_inv_tau(s, n);
  CK(cudaMemcpyAsync(m->dyn_dev, m->dyn_host, sizeof(dg::StepParams), cudaMemcpyHostToDevice,
                     m->stream));
  return DG_OK;
}

int denoise_impl(dg_model *m, int32_t *done) {
  CKR(begin_canvas(m));
  m->step += 1;
  CKR(put_step_params(m, m->step));
  const dg_model::StepGraph *used = nullptr;
  if (!m->eager_step_done) {
    CKR(step_launches(m));
    m->eager_step_done = true;
  } else {
    const auto key = std::make_pair(graph_key(m), m->prof_on ? 1 : 0);
    auto it = m->graphs.find(key);
    if (it == m->graphs.end()) {
      dg_model::StepGraph g;
      const int r = capture_step(m, &g);
      if (r != DG_OK) {
        for (auto &rec : g.recs) {
          cudaEventDestroy(rec.a);
          cudaEventDestroy(rec.b);
        }
        return r;
      }
      it = m->graphs.emplace(key, std::move(g)).first;
    }
    CK(cudaGraphLaunch(it->second.exec, m->stream));
    used = &it->second;
  }
  CK(cudaMemcpyAsync(m->done_host, m->done_dev, 2 * sizeof(int), cudaMemcpyDeviceToHost, m->stream));
  SYNC(m);
  m->host_syncs += 1;
  if (used) prof_collect_graph(m, *used);
  if (m->done_host[1])
    return device_fail(m->done_host[1]);
  m->canvas_done = m->done_host[0] != 0;
  if (done) *done = m->canvas_done ? 1 : 0;
  return DG_OK;
}

// Capture the canvas loop for the current prefix length: a graph holding one
// WHILE conditional node (condition 1 at launch) whose body is the step;
// the step's rule kernel clears the condition once the canvas is done.
int capture_loop(dg_model *m, dg_model::LoopGraph *lg) {
  cudaGraph_t graph = nullptr;
  CK(cudaGraphCreate(&graph, 0));
  cudaGraphConditionalHandle h;
  cudaError_t e = cudaGraphConditionalHandleCreate(&h, graph, 1, cudaGraphCondAssignDefault);
  cudaGraphNodeParams cp = {};
  cudaGraphNode_t node;
  if (e == cudaSuccess) {
    cp.type = cudaGraphNodeTypeConditional;
    cp.conditional.handle = h;
    cp.conditional.type = cudaGraphCondTypeWhile;
    cp.conditional.size = 1;
    e = cudaGraphAddNode(&node, graph, nullptr, nullptr, 0, &cp);
  }
  if (e == cudaSuccess)
    e = cudaStreamBeginCaptureToGraph(m->stream, cp.conditional.phGraph_out[0], nullptr, nullptr, 0,
                                      cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) {
    cudaGraphDestroy(graph);
    return fail(DG_ECUDA, "canvas loop graph: %s", cudaGetErrorString(e));
  }
  dg_model::StepGraph counts;  // launch counts of one iteration (no event nodes: profiling is off)
  m->capturing = &counts;
  m->loop_ctl = dg::LoopCtl{1, h, m->sc.temp_start, m->sc.temp_end, m->done_dev + 1};
  const int r = step_launches(m);
  m->loop_ctl = dg::LoopCtl{};
  m->capturing = nullptr;
  cudaGraph_t body = nullptr;
  e = cudaStreamEndCapture(m->stream, &body);
  if (r != DG_OK || e != cudaSuccess) {
    cudaGraphDestroy(graph);
    return r != DG_OK ? r : fail(DG_ECUDA, "canvas loop capture: %s", cudaGetErrorString(e));
  }
  e = cudaGraphInstantiate(&lg->exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return fail(DG_ECUDA, "canvas loop instantiation: %s", cudaGetErrorString(e));
  for (int i = 0; i < DG_K_CLASSES; ++i) lg->launches[i] = counts.launches[i];
  return DG_OK;
}

// Denoise the current canvas to the end.  With profiling off and the
// kernels' attributes set (one eager step done), every remaining step runs
// in one launch of the device-side loop, with a single synchronisation;
// otherwise step by step.
int denoise_canvas_impl(dg_model *m, int32_t *n_steps) {
  CKR(begin_canvas(m));
  const int start = m->step;
  if (m->prof_on || !m->eager_step_done) {
    int32_t done = 0;
    CKR(denoise_impl(m, &done));
    while (!done && m->prof_on) CKR(denoise_impl(m, &done));
    if (done) {
      if (n_steps) *n_steps = m->step - start;
      return DG_OK;
    }
  }
  auto it = m->loop_graphs.find(graph_key(m));
  if (it == m->loop_graphs.end()) {
    dg_model::LoopGraph lg;
    CKR(capture_loop(m, &lg));
    it = m->loop_graphs.emplace(graph_key(m), lg).first;
  }
  CKR(put_step_params(m, m->step + 1));
  CK(cudaGraphLaunch(it->second.exec, m->stream));
  CK(cudaMemcpyAsync(m->done_host, m->done_dev, 2 * sizeof(int), cudaMemcpyDeviceToHost, m->stream));
  CK(cudaMemcpyAsync(&m->dyn_host->step, &m->dyn_dev->step, sizeof(int), cudaMemcpyDeviceToHost, m->stream));
  SYNC(m);
  m->host_syncs += 1;
  if (m->done_host[1])
    return device_fail(m->done_host[1]);
  const int steps = m->dyn_host->step - start;  // the loop leaves dyn at its last step
  const int loop_steps = m->dyn_host->step - m->step;
  for (int i = 0; i < DG_K_CLASSES; ++i) m->prof_launches[i] += it->second.launches[i] * loop_steps;
  m->step = m->dyn_host->step;
  m->canvas_done = m->done_host[0] != 0;
  if (!m->canvas_done) return fail(DG_ECUDA, "the canvas loop ended before the canvas was done");
  if (n_steps) *n_steps = steps;
  return DG_OK;
}

int valid_tokens(const int32_t *ids, int C, int eos) {
  if (eos < 0) return C;
  for (int i = 0; i < C; ++i)
    if (ids[i] == eos) return i;
  return C;
}

// Finish the current canvas(es): ids to out_ids (host, B * C), C_k of each
// request to out_valid (host, B), then (append) the one KV-append forward of
// every request's canvas, each after its own prefix.
int commit_impl(dg_model *m, int32_t *out_ids, int32_t *out_valid, bool append) {
  if (!m->canvas_active || !m->canvas_done) return fail(DG_ESTATE, "canvas not finished");
  const int C = m->sc.canvas_len, T = m->B * C;
  std::vector<int32_t> ids(T);
  CK(cudaMemcpyAsync(ids.data(), m->x, sizeof(int) * T, cudaMemcpyDeviceToHost, m->stream));
  SYNC(m);
  if (out_ids) memcpy(out_ids, ids.data(), sizeof(int) * T);
  if (out_valid)
    for (int b = 0; b < m->B; ++b) out_valid[b] = valid_tokens(ids.data() + (size_t)b * C, C, m->sc.eos_id);
  if (append) {
    KL(DG_K_EMBED, 1, dg::embed_rows(m->h, m->embed, m->x, T, m->cfg.d_model, m->stream));
    CKR(run_layers(m, T, canvas_rows(m), m->page_table, m->sc.commit_causal ? 1 : 0, true));
    CKR(sync_check(m));
    for (int b = 0; b < m->B; ++b) m->prefix_lens[b] += C;
    m->prefix_len = m->prefix_lens[0];
    m->canvas_index += 1;
    m->canvas_active = m->canvas_done = false;
  }
  return DG_OK;
}

// Per-request step counts of the canvases just finished (B > 1: the step at
// which each request's canvas finished; B = 1: the steps taken).
int read_request_steps(dg_model *m, std::vector<int> &nk) {
  nk.assign(m->B, m->step);
  if (m->B > 1) {
    CK(cudaMemcpyAsync(nk.data(), m->req_nk, sizeof(int) * m->B, cudaMemcpyDeviceToHost, m->stream));
    SYNC(m);
  }
  return DG_OK;
}

int single_only(dg_model *m) {
  if (m->B != 1) return fail(DG_EINVAL, "the model holds %d requests: use the batch calls", m->B);
  return DG_OK;
}

}  // namespace

extern "C" {

const char *dg_last_error(void) { return g_err.c_str(); }

int dg_init_model(const dg_config *cfg, const dg_sampler_config *scfg, const void *const *weights,
                  void *cuda_stream, dg_model **out) {
  if (!out) return fail(DG_EINVAL, "null out");
  *out = nullptr;
  CKR(validate(cfg, scfg));
  dg_model *m = new dg_model();
  m->cfg = *cfg;
  m->sc = *scfg;
  m->B = cfg->max_requests > 1 ? cfg->max_requests : 1;
  m->prompt_lens.assign(m->B, 0);
  m->prefix_lens.assign(m->B, 0);
  if (const char *f = getenv("DG_FAULT_ALLOC")) m->fail_alloc_at = atoi(f);
  if (const char *f = getenv("DG_FAULT")) {  // alloc:n | badcall:n | kvfull
    if (!strncmp(f, "alloc:", 6)) m->fail_alloc_at = atoi(f + 6);
    else if (!strncmp(f, "badcall:", 8)) m->fail_launch_at = atoi(f + 8);
    else if (!strcmp(f, "kvfull")) m->fault_kvfull = true;
  }
  if (cuda_stream) {
    m->stream = (cudaStream_t)cuda_stream;
  } else {
    if (cudaStreamCreateWithFlags(&m->stream, cudaStreamNonBlocking) != cudaSuccess) {
      cudaGetLastError();
      delete m;
      return fail(DG_ECUDA, "cudaStreamCreate failed");
    }
    m->own_stream = true;
  }
  int r = alloc_model(m, weights);
  if (r == DG_OK && !weights) r = fill_model_weights(m);
  if (r == DG_OK && cfg->expert_fp8) r = quantize_expert_weights(m);
  if (r == DG_OK) {
    cudaError_t e = dg::rope_table(m->cos_t, m->sin_t, cfg->max_context, cfg->head_dim,
                                   cfg->rope_base, m->stream);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(m->page_table, m->page_table_host.data(), sizeof(int) * m->n_pages,
                          cudaMemcpyHostToDevice, m->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(m->stream);
    if (e != cudaSuccess) r = fail(DG_ECUDA, "model set-up: %s", cudaGetErrorString(e));
  }
  if (r != DG_OK) {
    std::string keep = g_err;
    dg_free_model(m);
    g_err = keep;
    return r;
  }
  *out = m;
  return DG_OK;
}

void dg_free_model(dg_model *m) {
  if (!m) return;
  if (m->stream) cudaStreamSynchronize(m->stream);
  prof_collect(m);
  destroy_graphs(m);
  for (cudaEvent_t e : m->prof_free) cudaEventDestroy(e);
  for (void *p : m->allocs) cudaFree(p);
  if (m->done_host) cudaFreeHost(m->done_host);
  if (m->dyn_host) cudaFreeHost(m->dyn_host);
  if (m->own_stream) cudaStreamDestroy(m->stream);
  delete m;
}

int dg_prefill(dg_model *m, const int32_t *prompt_ids, int32_t n) {
  CKR(check_model(m));
  CKR(single_only(m));
  return prefill_impl(m, prompt_ids, n);
}

int dg_denoise_step(dg_model *m, int32_t *done) {
  CKR(check_model(m));
  CKR(single_only(m));
  return denoise_impl(m, done);
}

int dg_denoise_canvas(dg_model *m, int32_t *n_steps) {
  CKR(check_model(m));
  CKR(single_only(m));
  return denoise_canvas_impl(m, n_steps);
}

int dg_commit_canvas(dg_model *m, int32_t *out_ids, int32_t *out_valid) {
  CKR(check_model(m));
  CKR(single_only(m));
  return commit_impl(m, out_ids, out_valid, true);
}

int dg_prefill_batch(dg_model *m, const int32_t *const *prompts, const int32_t *lens) {
  CKR(check_model(m));
  if (!prompts || !lens) return fail(DG_EINVAL, "null prompts");
  for (int b = 0; b < m->B; ++b) CKR(check_prompt(m, prompts[b], lens[b]));
  for (int b = 0; b < m->B; ++b) CKR(encode_prompt(m, b, prompts[b], lens[b]));
  m->prompt_lens.assign(lens, lens + m->B);
  reset_generation(m);
  return DG_OK;
}

int dg_denoise_canvas_batch(dg_model *m, int32_t *n_steps) {
  CKR(check_model(m));
  int32_t n = 0;
  CKR(denoise_canvas_impl(m, &n));
  std::vector<int> nk;
  CKR(read_request_steps(m, nk));
  if (n_steps) memcpy(n_steps, nk.data(), sizeof(int) * m->B);
  return DG_OK;
}

int dg_commit_canvas_batch(dg_model *m, int32_t *out_ids, int32_t *out_valid) {
  CKR(check_model(m));
  return commit_impl(m, out_ids, out_valid, true);
}

int dg_generate_batch(dg_model *m, const int32_t *const *prompts, const int32_t *lens, int32_t K_max,
                      int32_t *out_ids, dg_stats *stats) {
  CKR(check_model(m));
  if (K_max < 1 || !out_ids) return fail(DG_EINVAL, "K_max >= 1 and out_ids required");
  const int B = m->B, C = m->sc.canvas_len;
  const double t0 = now_s();
  CKR(dg_prefill_batch(m, prompts, lens));
  const double t1 = now_s();
  std::vector<std::vector<int>> Ns(B), Cs(B);
  std::vector<char> active(B, 1);
  std::vector<int32_t> ids((size_t)B * C), valid(B);
  const int64_t syncs0 = m->host_syncs;
  for (int k = 0; k < K_max; ++k) {
    int32_t n = 0;
    CKR(denoise_canvas_impl(m, &n));
    std::vector<int> nk;
    CKR(read_request_steps(m, nk));
    CKR(commit_impl(m, ids.data(), valid.data(), false));
    bool any = false;
    for (int b = 0; b < B; ++b) {
      if (!active[b]) continue;
      memcpy(out_ids + ((size_t)b * K_max + k) * C, ids.data() + (size_t)b * C, sizeof(int32_t) * C);
      Ns[b].push_back(nk[b]);
      Cs[b].push_back(valid[b]);
      if (valid[b] < C) active[b] = 0;  // its generation ends with the canvas holding its first EOS
      any = any || active[b];
    }
    if (!any || k == K_max - 1) break;
    CKR(commit_impl(m, nullptr, nullptr, true));
  }
  const double t2 = now_s();
  for (int b = 0; stats && b < B; ++b) {
    dg_stats &st = stats[b];
    const int K = (int)Ns[b].size();
    long long tok = 0, steps = 0, wsum = 0;
    for (int i = 0; i < K; ++i) {
      tok += Cs[b][i];
      steps += Ns[b][i];
      wsum += (long long)Ns[b][i] * Cs[b][i];
      if (st.N_k) st.N_k[i] = Ns[b][i];
      if (st.C_k) st.C_k[i] = Cs[b][i];
    }
    st.K = K;
    st.total_tokens = (int)tok;
    st.total_steps = (int)steps;
    st.n_forwards = (int)(steps + K - 1);
    st.effective_steps = tok ? (double)wsum / (double)tok : 0.0;
    st.tpf = (double)tok / (double)(steps + K - 1);
    st.prefill_seconds = t1 - t0;
    st.decode_seconds = t2 - t1;
    st.steps_per_s = t2 > t1 ? (double)steps / (t2 - t1) : 0.0;
    st.tokens_per_s = t2 > t1 ? (double)tok / (t2 - t1) : 0.0;
    st.canvas_loop_syncs = (int32_t)(m->host_syncs - syncs0);
  }
  return DG_OK;
}

int dg_generate(dg_model *m, const int32_t *prompt, int32_t n_prompt, int32_t K_max,
                int32_t *out_ids, dg_stats *stats) {
  CKR(check_model(m));
  CKR(single_only(m));
  if (K_max < 1 || !out_ids) return fail(DG_EINVAL, "K_max >= 1 and out_ids required");
  const int C = m->sc.canvas_len;
  const double t0 = now_s();
  CKR(prefill_impl(m, prompt, n_prompt));
  const double t1 = now_s();
  std::vector<int> Ns, Cs;
  const int64_t syncs0 = m->host_syncs;
  for (int k = 0; k < K_max; ++k) {
    int n = 0;
    CKR(denoise_canvas_impl(m, &n));
    int valid = 0;
    const bool last = (k == K_max - 1);
    CKR(commit_impl(m, out_ids + (size_t)k * C, &valid, false));
    Ns.push_back(n);
    Cs.push_back(valid);
    if (valid < C || last) break;
    CKR(commit_impl(m, nullptr, nullptr, true));
  }
  const double t2 = now_s();
  if (stats) {
    const int K = (int)Ns.size();
    long long tok = 0, steps = 0, wsum = 0;
    for (int i = 0; i < K; ++i) {
      tok += Cs[i];
      steps += Ns[i];
      wsum += (long long)Ns[i] * Cs[i];
      if (stats->N_k) stats->N_k[i] = Ns[i];
      if (stats->C_k) stats->C_k[i] = Cs[i];
    }
    stats->K = K;
    stats->total_tokens = (int)tok;
    stats->total_steps = (int)steps;
    stats->n_forwards = (int)(steps + K - 1);
    stats->effective_steps = tok ? (double)wsum / (double)tok : 0.0;
    stats->tpf = (double)tok / (double)(steps + K - 1);
    stats->prefill_seconds = t1 - t0;
    stats->decode_seconds = t2 - t1;
    stats->steps_per_s = t2 > t1 ? (double)steps / (t2 - t1) : 0.0;
    stats->canvas_loop_syncs = (int32_t)(m->host_syncs - syncs0);
    stats->tokens_per_s = t2 > t1 ? (double)tok / (t2 - t1) : 0.0;
  }
  return DG_OK;
}

int dg_set_sampler(dg_model *m, const dg_sampler_config *scfg) {
  CKR(check_model(m));
  CKR(validate(&m->cfg, scfg));
  if (scfg->canvas_len != m->sc.canvas_len) return fail(DG_EINVAL, "canvas_len is fixed at init");
  const dg_sampler_config &o = m->sc;
  if (scfg->budget_N != o.budget_N || scfg->stable_steps != o.stable_steps ||
      scfg->adaptive != o.adaptive || scfg->conf_threshold != o.conf_threshold ||
      scfg->temp_start != o.temp_start || scfg->temp_end != o.temp_end) {
    CK(cudaStreamSynchronize(m->stream));
    destroy_graphs(m);  // captured steps hold the old rule constants
  }
  m->sc = *scfg;  // the sample seed is read per step from device memory
  return DG_OK;
}

int dg_rewind(dg_model *m, int32_t n_prefix) {
  CKR(check_model(m));
  CKR(single_only(m));
  if (!m->prefilled) return fail(DG_ESTATE, "nothing cached");
  if (n_prefix < m->prompt_len || n_prefix > m->prefix_len ||
      (n_prefix - m->prompt_len) % m->sc.canvas_len)
    return fail(DG_EINVAL, "n_prefix must be the prompt plus whole committed canvases");
  m->prefix_len = m->prefix_lens[0] = n_prefix;
  m->canvas_index = (n_prefix - m->prompt_len) / m->sc.canvas_len;
  m->canvas_active = m->canvas_done = false;
  return DG_OK;
}

int dg_read_canvas(dg_model *m, int32_t *ids, uint8_t *committed, int32_t *last_argmax,
                   int32_t *stable, int32_t *step, int32_t *canvas_index, int32_t *prefix_len) {
  CKR(check_model(m));
  const int C = m->sc.canvas_len;
  if (ids) CK(cudaMemcpyAsync(ids, m->x, sizeof(int) * C, cudaMemcpyDeviceToHost, m->stream));
  if (committed) CK(cudaMemcpyAsync(committed, m->committed, C, cudaMemcpyDeviceToHost, m->stream));
  if (last_argmax)
    CK(cudaMemcpyAsync(last_argmax, m->last, sizeof(int) * C, cudaMemcpyDeviceToHost, m->stream));
  if (stable) CK(cudaMemcpyAsync(stable, m->stable, sizeof(int) * C, cudaMemcpyDeviceToHost, m->stream));
  SYNC(m);
  if (step) *step = m->step;
  if (canvas_index) *canvas_index = m->canvas_index;
  if (prefix_len) *prefix_len = m->prefix_len;
  return DG_OK;
}

int dg_write_canvas(dg_model *m, const int32_t *ids, const uint8_t *committed,
                    const int32_t *last_argmax, const int32_t *stable, int32_t step,
                    int32_t canvas_index) {
  CKR(check_model(m));
  CKR(single_only(m));
  if (!m->prefilled) return fail(DG_ESTATE, "dg_prefill must come first");
  if (!ids || !committed || !last_argmax || !stable || step < 0 || canvas_index < 0)
    return fail(DG_EINVAL, "all state arrays are required");
  const int C = m->sc.canvas_len;
  for (int i = 0; i < C; ++i)
    if (ids[i] < 0 || ids[i] >= m->cfg.vocab) return fail(DG_EINVAL, "id out of range");
  CK(cudaMemcpyAsync(m->x, ids, sizeof(int) * C, cudaMemcpyHostToDevice, m->stream));
  CK(cudaMemcpyAsync(m->committed, committed, C, cudaMemcpyHostToDevice, m->stream));
  CK(cudaMemcpyAsync(m->last, last_argmax, sizeof(int) * C, cudaMemcpyHostToDevice, m->stream));
  CK(cudaMemcpyAsync(m->stable, stable, sizeof(int) * C, cudaMemcpyHostToDevice, m->stream));
  SYNC(m);
  m->step = step;
  m->canvas_index = canvas_index;
  m->canvas_active = true;
  m->canvas_done = false;
  return DG_OK;
}

int dg_read_step_outputs(dg_model *m, int32_t *argmax, float *conf, int32_t *gumbel) {
  CKR(check_model(m));
  const int C = m->sc.canvas_len;
  if (argmax) CK(cudaMemcpyAsync(argmax, m->argmax, sizeof(int) * C, cudaMemcpyDeviceToHost, m->stream));
  if (conf) CK(cudaMemcpyAsync(conf, m->conf, sizeof(float) * C, cudaMemcpyDeviceToHost, m->stream));
  if (gumbel) CK(cudaMemcpyAsync(gumbel, m->gumbel, sizeof(int) * C, cudaMemcpyDeviceToHost, m->stream));
  SYNC(m);
  return DG_OK;
}

int dg_canvas_logits(dg_model *m, float *logits_dev) {
  CKR(check_model(m));
  CKR(single_only(m));
  if (!logits_dev) return fail(DG_EINVAL, "null logits");
  CKR(begin_canvas(m));
  CKR(canvas_forward(m));
  const dg_config &c = m->cfg;
  KL(DG_K_LM_HEAD, 1,
     dg::gemm_lm_head_logits(m->xn, m->xn_lo, m->lm_head, m->sc.canvas_len, c.d_model, c.vocab,
                             logits_dev, m->done_dev + 1, m->stream));
  SYNC(m);
  return DG_OK;
}

int dg_read_kv(dg_model *m, int32_t layer, int32_t pos0, int32_t n, uint16_t *k_out,
               uint16_t *v_out) {
  CKR(check_model(m));
  const dg_config &c = m->cfg;
  if (layer < 0 || layer >= c.n_layers || pos0 < 0 || n < 0 || pos0 + n > m->n_pages * c.page_size)
    return fail(DG_EINVAL, "bad range");
  const int hd = c.head_dim, Hkv = c.n_kv_heads, pg = c.page_size;
  if (n == 0) return DG_OK;
  // whole pages to the host, then slot rows out of the pool's tiled order
  // (element f of slot s: sub-block f / 64, row s, chunk ((f % 64) / 8) ^ (s % 8))
  const size_t page_elems = (size_t)Hkv * pg * hd;
  std::vector<uint16_t> kb(page_elems), vb(page_elems);
  for (int pl = pos0 / pg; pl <= (pos0 + n - 1) / pg; ++pl) {
    const size_t off = (size_t)m->page_table_host[pl] * page_elems;
    if (k_out) CK(cudaMemcpyAsync(kb.data(), m->kpool(layer) + off, page_elems * 2, cudaMemcpyDeviceToHost, m->stream));
    if (v_out) CK(cudaMemcpyAsync(vb.data(), m->vpool(layer) + off, page_elems * 2, cudaMemcpyDeviceToHost, m->stream));
    SYNC(m);
    const int t0 = pl * pg > pos0 ? pl * pg : pos0, t1 = (pl + 1) * pg < pos0 + n ? (pl + 1) * pg : pos0 + n;
    for (int p = t0; p < t1; ++p) {
      const int sl = p % pg;
      for (int h = 0; h < Hkv; ++h)
        for (int f = 0; f < hd; ++f) {
          const size_t src = (size_t)h * pg * hd + (size_t)(f / 64) * pg * 64 + (size_t)sl * 64 +
                             ((((f % 64) / 8) ^ (sl % 8)) * 8) + f % 8;
          const size_t dst = ((size_t)(p - pos0) * Hkv + h) * hd + f;
          if (k_out) k_out[dst] = kb[src];
          if (v_out) v_out[dst] = vb[src];
        }
    }
  }
  return DG_OK;
}

int dg_read_routing(dg_model *m, int32_t layer, int32_t *ids, int32_t max_rows, int32_t *n_rows) {
  CKR(check_model(m));
  if (layer < 0 || layer >= m->cfg.n_layers) return fail(DG_EINVAL, "bad layer");
  const int rows = m->routing_rows[layer];
  if (n_rows) *n_rows = rows;
  if (ids) {
    const int n = rows < max_rows ? rows : max_rows;
    CK(cudaMemcpyAsync(ids, m->topk + (size_t)layer * m->Tmax * m->cfg.top_k,
                       sizeof(int) * (size_t)n * m->cfg.top_k, cudaMemcpyDeviceToHost, m->stream));
    SYNC(m);
  }
  return DG_OK;
}

int dg_read_moe_input(dg_model *m, uint16_t *rows, int32_t max_rows, int32_t *n_rows, int32_t *layer) {
  CKR(check_model(m));
  if (n_rows) *n_rows = m->moe_input_rows;
  if (layer) *layer = m->moe_input_layer;
  if (rows && m->moe_input_rows > 0) {
    const int n = m->moe_input_rows < max_rows ? m->moe_input_rows : max_rows;
    CK(cudaMemcpyAsync(rows, m->xn, sizeof(uint16_t) * (size_t)n * m->cfg.d_model, cudaMemcpyDeviceToHost,
                       m->stream));
    SYNC(m);
  }
  return DG_OK;
}

int dg_read_page_table(dg_model *m, int32_t *table, int32_t max_entries, int32_t *n_pages) {
  CKR(check_model(m));
  const int used = dg::ceil_div(m->prefix_len + (m->canvas_active ? m->sc.canvas_len : 0),
                                m->cfg.page_size);
  if (n_pages) *n_pages = used;
  if (table) {
    std::vector<int> dev(m->n_pages);
    CK(cudaMemcpyAsync(dev.data(), m->page_table, sizeof(int) * m->n_pages, cudaMemcpyDeviceToHost,
                       m->stream));
    SYNC(m);
    for (int i = 0; i < used && i < max_entries; ++i) table[i] = dev[i];
  }
  return DG_OK;
}

int dg_get_weight(dg_model *m, int32_t which, int32_t layer, void **dev_ptr, size_t *bytes) {
  CKR(check_model(m));
  const dg_config &c = m->cfg;
  const size_t d = c.d_model, qd = (size_t)c.n_q_heads * c.head_dim,
               kd = (size_t)c.n_kv_heads * c.head_dim;
  const size_t E = c.n_experts, F = c.d_ff;
  const bool per_layer = which >= DG_W_WQKV;
  if (per_layer && (layer < 0 || layer >= c.n_layers)) return fail(DG_EINVAL, "bad layer");
  void *p = nullptr;
  size_t b = 0;
  switch (which) {
    case DG_W_EMBED: p = m->embed; b = (size_t)c.vocab * d * 2; break;
    case DG_W_LM_HEAD: p = m->lm_head; b = (size_t)c.vocab * d * 2; break;
    case DG_W_FINAL_NORM: p = m->final_norm; b = d * 4; break;
    case DG_W_WQKV: p = m->layers[layer].wqkv; b = (qd + 2 * kd) * d * 2; break;
    case DG_W_WO: p = m->layers[layer].wo; b = d * qd * 2; break;
    case DG_W_ROUTER: p = m->layers[layer].wr; b = E * d * 2; break;
    case DG_W_GATE_UP: p = m->layers[layer].wgu; b = E * 2 * F * d * 2; break;
    case DG_W_DOWN: p = m->layers[layer].wd; b = E * d * F * 2; break;
    case DG_W_ATTN_NORM: p = m->layers[layer].attn_norm; b = d * 4; break;
    case DG_W_MOE_NORM: p = m->layers[layer].moe_norm; b = d * 4; break;
    default: return fail(DG_EINVAL, "unknown weight %d", which);
  }
  if (dev_ptr) *dev_ptr = p;
  if (bytes) *bytes = b;
  return DG_OK;
}

const char *dg_kernel_class_name(int32_t cls) {
  static const char *names[DG_K_CLASSES] = {
      "embed", "rmsnorm", "qkv_rope", "attention", "o_proj", "route",
      "expert_ffn", "combine", "lm_head", "sampler_merge", "sampler_rule",
      "canvas_init"};
  return (cls >= 0 && cls < DG_K_CLASSES) ? names[cls] : "";
}

int dg_profile(dg_model *m, int32_t enable) {
  CKR(check_model(m));
  SYNC(m);
  m->prof_on = enable == 1;
  if (enable != 0) {
    for (int i = 0; i < DG_K_CLASSES; ++i) {
      m->prof_ms[i] = 0.0;
      m->prof_launches[i] = 0;
    }
    CK(cudaMemsetAsync(m->moe_stats, 0, 2 * sizeof(unsigned long long), m->stream));
    SYNC(m);
  }
  return DG_OK;
}

int dg_profile_experts(dg_model *m, int64_t *experts_touched, int64_t *rows_routed) {
  CKR(check_model(m));
  unsigned long long v[2] = {0, 0};
  CK(cudaMemcpyAsync(v, m->moe_stats, sizeof(v), cudaMemcpyDeviceToHost, m->stream));
  SYNC(m);
  if (experts_touched) *experts_touched = (int64_t)v[0];
  if (rows_routed) *rows_routed = (int64_t)v[1];
  return DG_OK;
}

int dg_profile_read(dg_model *m, double *ms, int64_t *launches) {
  CKR(check_model(m));
  SYNC(m);
  for (int i = 0; i < DG_K_CLASSES; ++i) {
    if (ms) ms[i] = m->prof_ms[i];
    if (launches) launches[i] = m->prof_launches[i];
  }
  return DG_OK;
}

// ---- kernel-level entry points ----------------------------------------------

}  // extern "C"

namespace {

// Status words of the kernel-level entry points, one set per device that loads
// the library: a bounded device-side wait that gives up writes its code to
// [0], and the attention writes 39 to [1] for a page index outside the pools.  It is a
// file-scope device array rather than an allocation, so that the entry points
// that must not allocate can use it too; it is zero when the library is
// loaded, sticky (a later kernel that sees it set skips its waits), and read
// and cleared by dg_op_status.  Calls that overlap on the GPU share it.
static __device__ __align__(256) int g_op_status[64];

std::mutex g_status_mu;
int *g_status_ptr[64];

// Address of g_op_status on the current device.  In host code the array's
// name is only a stand-in, so the address is looked up once per device, with
// that device current, by the first kernel-level call made on it.
int op_status_ptr(int **out) {
  int dev = 0;
  CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(DG_EINVAL, "device %d: only devices 0-63 are supported", dev);
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (!g_status_ptr[dev]) {
    void *p = nullptr;
    CK(cudaGetSymbolAddress(&p, g_op_status));
    g_status_ptr[dev] = (int *)p;
  }
  *out = g_status_ptr[dev];
  return DG_OK;
}

int check_attention_args(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                         const int32_t *page_table, const uint16_t *out, int32_t n_prefix,
                         int32_t n_new, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                         int32_t page_size, int32_t n_pages) {
  if (!q || !k_pool || !v_pool || !page_table || !out) return fail(DG_EINVAL, "null pointer");
  if (n_prefix < 0 || n_new < 0 || n_kv_heads < 1 || n_q_heads % n_kv_heads ||
      (head_dim != 64 && head_dim != 128) || page_size < 64 || page_size % 64 || n_pages < 1)
    return fail(DG_EINVAL, "unsupported attention shape");
  if ((int64_t)n_pages * page_size < (int64_t)n_prefix + n_new)
    return fail(DG_EINVAL, "%d pages of %d tokens cannot hold %d keys", n_pages, page_size, n_prefix + n_new);
  return DG_OK;
}

}  // namespace

extern "C" {

int dg_op_status(void *stream) {
  int *st = nullptr;
  CKR(op_status_ptr(&st));
  CK(cudaStreamSynchronize((cudaStream_t)stream));
  int v[2] = {0, 0};
  CK(cudaMemcpy(v, st, sizeof(v), cudaMemcpyDeviceToHost));
  if (v[0] == 0 && v[1] == 0) return DG_OK;
  CK(cudaMemset(st, 0, sizeof(v)));
  if (v[0]) return device_fail(v[0]);
  return fail(DG_EINVAL, "a page table entry was outside the pools (its keys were skipped)");
}


int dg_op_fill_weights(uint16_t *dst, uint64_t n, uint64_t seed, uint32_t tensor_id, uint64_t e0,
                       float std_dev, void *stream) {
  if (!dst && n) return fail(DG_EINVAL, "null dst");
  CK(dg::fill_weights((bf16 *)dst, n, seed, tensor_id, e0, std_dev, (cudaStream_t)stream));
  return DG_OK;
}

size_t dg_op_attention_workspace_bytes(int32_t n_prefix, int32_t n_new, int32_t n_q_heads,
                                       int32_t n_kv_heads, int32_t head_dim) {
  if (n_kv_heads < 1 || n_new < 0 || n_prefix < 0) return 0;
  dg::AttnShape as{n_prefix, n_new, n_q_heads, n_kv_heads, head_dim, 64, 0};
  return dg::attention_workspace_bytes(as);
}

int dg_op_wait_selftest(int64_t limit_cycles, void *stream) {
  if (limit_cycles < 1 || limit_cycles > (int64_t)1 << 31) return fail(DG_EINVAL, "limit_cycles out of range");
  int *status = nullptr;
  CKR(op_status_ptr(&status));
  CK(dg::bounded_wait_selftest(status, (long long)limit_cycles, (cudaStream_t)stream));
  return DG_OK;
}

int dg_op_canvas_attention(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                           const int32_t *page_table, int32_t n_prefix, int32_t n_new,
                           int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                           int32_t page_size, int32_t n_pages, int32_t causal, uint16_t *out,
                           void *workspace, size_t workspace_bytes, void *stream) {
  CKR(check_attention_args(q, k_pool, v_pool, page_table, out, n_prefix, n_new, n_q_heads, n_kv_heads,
                           head_dim, page_size, n_pages));
  dg::AttnShape as{n_prefix, n_new, n_q_heads, n_kv_heads, head_dim, page_size, causal ? 1 : 0, n_pages};
  if (workspace_bytes < dg::attention_workspace_bytes(as)) return fail(DG_EINVAL, "workspace too small");
  int *status = nullptr;
  CKR(op_status_ptr(&status));
  CK(dg::attention((const bf16 *)q, (const bf16 *)k_pool, (const bf16 *)v_pool, page_table, as,
                   (bf16 *)out, workspace, workspace_bytes, (cudaStream_t)stream, status));
  return DG_OK;
}

int dg_op_canvas_attention_noalloc(const uint16_t *q, const uint16_t *k_pool,
                                   const uint16_t *v_pool, const int32_t *page_table,
                                   int32_t n_prefix, int32_t n_new, int32_t n_q_heads,
                                   int32_t n_kv_heads, int32_t head_dim, int32_t page_size,
                                   int32_t n_pages, int32_t causal, uint16_t *out, void *stream) {
  CKR(check_attention_args(q, k_pool, v_pool, page_table, out, n_prefix, n_new, n_q_heads, n_kv_heads,
                           head_dim, page_size, n_pages));
  dg::AttnShape as{n_prefix, n_new, n_q_heads, n_kv_heads, head_dim, page_size, causal ? 1 : 0, n_pages};
  int *status = nullptr;  // the library's status array: no device memory of the caller's or ours
  CKR(op_status_ptr(&status));
  CK(dg::attention((const bf16 *)q, (const bf16 *)k_pool, (const bf16 *)v_pool, page_table, as,
                   (bf16 *)out, nullptr, 0, (cudaStream_t)stream, status));
  return DG_OK;
}

}  // extern "C"

namespace {
struct MoeWs {
  int *offs, *gcount, *slot_row, *work, *n_work;
  bf16 *act, *x_tiles;
  bf16 *y_rows;
  int *bar;
  float *part;
  size_t bytes;
  int max_work;
};
MoeWs moe_layout(void *base, int T, int d, int E, int k, int F) {
  MoeWs w{};
  unsigned char *p = (unsigned char *)base;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    void *r = p ? p + off : nullptr;
    off += (bytes + 255) & ~(size_t)255;
    return r;
  };
  w.max_work = (int)dg::moe_max_work(T, k, E, dg::kExpertTileRows);
  w.offs = (int *)take((size_t)(E + 1) * 4);
  w.gcount = (int *)take(dg::moe_group_count_ints(T, E) * 4);
  w.slot_row = (int *)take((size_t)T * k * 4);
  w.work = (int *)take(dg::moe_work_ints(T, k, E, dg::kExpertTileRows) * 4);
  w.n_work = (int *)take(4);
  w.act = (bf16 *)take(dg::moe_item_tile_elems(w.max_work, F) * 2);
  w.x_tiles = (bf16 *)take(dg::moe_item_tile_elems(w.max_work, d) * 2);
  w.y_rows = (bf16 *)take((size_t)T * k * d * 2);
  w.bar = (int *)take(dg::kGridBarInts * 4);
  w.part = (float *)take(dg::moe_ffn_part_slots() * dg::kFfnPartSlotBytes);
  w.bytes = off;
  return w;
}
}  // namespace

extern "C" {

size_t dg_op_moe_workspace_bytes(int32_t T, int32_t d, int32_t n_experts, int32_t top_k,
                                 int32_t d_ff) {
  if (T < 0 || d < 1 || n_experts < 1 || top_k < 1 || d_ff < 1) return 0;
  return moe_layout(nullptr, T, d, n_experts, top_k, d_ff).bytes;
}

int dg_op_moe(const uint16_t *xn, const uint16_t *w_router, const uint16_t *w_gate_up,
              const uint16_t *w_down, int32_t T, int32_t d, int32_t n_experts, int32_t top_k,
              int32_t d_ff, float *y, int32_t *expert_ids, float *gates, void *workspace,
              size_t workspace_bytes, void *stream) {
  if (!xn || !w_router || !w_gate_up || !w_down || !y || !expert_ids || !gates || !workspace)
    return fail(DG_EINVAL, "null pointer");
  if (T < 1 || d % 64 || d_ff % 64 || n_experts < 1 || n_experts > 256 || top_k < 1 ||
      top_k > 16 || top_k > n_experts)
    return fail(DG_EINVAL, "unsupported MoE shape");
  MoeWs w = moe_layout(workspace, T, d, n_experts, top_k, d_ff);
  if (workspace_bytes < w.bytes) return fail(DG_EINVAL, "workspace too small");
  cudaStream_t st = (cudaStream_t)stream;
  int *status = nullptr;
  CKR(op_status_ptr(&status));
  CK(cudaMemsetAsync(w.bar, 0, dg::kGridBarInts * sizeof(int), st));
  CK(dg::moe_route_scatter(nullptr, nullptr, 0.0f, const_cast<bf16 *>((const bf16 *)xn), (const bf16 *)w_router, T,
                           d, n_experts, top_k, expert_ids, gates, w.slot_row, w.gcount, w.x_tiles, w.offs, w.work,
                           w.n_work, w.max_work, w.bar, status, st));
  const int rows = T * top_k;
  CK(dg::moe_ffn(w.x_tiles, rows, (const bf16 *)w_gate_up, (const bf16 *)w_down, w.offs, w.work, w.n_work,
                 w.max_work, n_experts, d, d_ff, w.act, w.y_rows, status, st, nullptr, w.part,
                 (int)dg::moe_ffn_part_slots()));
  CK(dg::moe_combine(y, w.y_rows, gates, w.slot_row, T, top_k, d, false, st));
  return DG_OK;
}

int dg_op_fill_moe_weights(uint16_t *w_router, uint16_t *w_gate_up, uint16_t *w_down, int32_t d,
                           int32_t n_experts, int32_t d_ff, int32_t layer, uint64_t seed,
                           float std_dev, void *stream) {
  if (!w_router || !w_gate_up || !w_down || d_ff % 64 || layer < 0) return fail(DG_EINVAL, "bad arguments");
  CK(dg::fill_moe_weights((bf16 *)w_router, (bf16 *)w_gate_up, (bf16 *)w_down, d, n_experts, d_ff,
                          layer, seed, std_dev, (cudaStream_t)stream));
  return DG_OK;
}

int dg_op_lm_head_partials(const uint16_t *xn, const uint16_t *xn_lo, const uint16_t *w_out,
                           int32_t rows, int32_t d, int32_t V, uint64_t sample_seed,
                           int32_t canvas, int32_t step, float inv_tau, void *partials,
                           float *logits, void *stream) {
  if (!xn || !w_out || !partials || rows < 1 || d % 64 || V % 256 || V < 256 || !(inv_tau > 0.0f))
    return fail(DG_EINVAL, "bad arguments");
  int *status = nullptr;
  CKR(op_status_ptr(&status));
  CK(dg::gemm_lm_head_partials((const bf16 *)xn, (const bf16 *)xn_lo, (const bf16 *)w_out, rows, d, V,
                               sample_seed, canvas, step, inv_tau, partials, status,
                               (cudaStream_t)stream, nullptr, logits));
  return DG_OK;
}

int dg_op_logits_partials(const float *logits, int32_t rows, int32_t V, uint64_t sample_seed,
                          int32_t canvas, int32_t step, float inv_tau, void *partials,
                          void *stream) {
  if (!logits || !partials || rows < 1 || V % 256 || V < 256 || !(inv_tau > 0.0f))
    return fail(DG_EINVAL, "bad arguments");
  CK(dg::logits_partials(logits, rows, V, sample_seed, canvas, step, inv_tau, partials,
                         (cudaStream_t)stream));
  return DG_OK;
}

int dg_op_fill_tiled_weights(uint16_t *dst, int32_t rows, int32_t cols, uint64_t seed,
                             uint32_t tensor_id, float std_dev, void *stream) {
  if (!dst || rows < 1 || cols < 64 || cols % 64) return fail(DG_EINVAL, "bad arguments");
  CK(dg::fill_tiled_weights((bf16 *)dst, rows, cols, rows, rows, tensor_id, tensor_id, tensor_id, seed, std_dev,
                            (cudaStream_t)stream));
  return DG_OK;
}

int dg_op_gumbel_noise(const uint32_t *words, float *out, uint64_t n, void *stream) {
  if ((!words || !out) && n) return fail(DG_EINVAL, "null pointer");
  CK(dg::gumbel_noise(words, out, (size_t)n, (cudaStream_t)stream));
  return DG_OK;
}

int dg_op_quantize_rows_e4m3(const uint16_t *src, int32_t n_mat, int32_t rows, int32_t cols, uint8_t *dst,
                             int32_t *exps, void *stream) {
  if (n_mat < 0 || rows < 0 || cols < 128 || cols % 128) return fail(DG_EINVAL, "cols must be a positive multiple of 128");
  if ((!src || !dst || !exps) && n_mat && rows) return fail(DG_EINVAL, "null pointer");
  CK(dg::quantize_rows_e4m3((const bf16 *)src, dst, exps, n_mat, rows, cols, (cudaStream_t)stream));
  return DG_OK;
}

int dg_op_sampler_update(const void *partials, int32_t C, int32_t V, int32_t step,
                         const dg_sampler_config *scfg, int32_t *x, uint8_t *committed,
                         int32_t *last_argmax, int32_t *stable, int32_t *argmax, float *conf,
                         int32_t *gumbel, int32_t *done_dev, void *stream) {
  if (!partials || !scfg || !x || !committed || !last_argmax || !stable || !argmax || !conf ||
      !gumbel || !done_dev || C < 1 || C > 1024 || V % 256 || V < 256 || step < 1)
    return fail(DG_EINVAL, "bad arguments");
  cudaStream_t st = (cudaStream_t)stream;
  CK(dg::sampler_merge(partials, C, V, argmax, conf, gumbel, st));
  CK(dg::sampler_rule(argmax, conf, gumbel, C, step, scfg->budget_N, scfg->stable_steps,
                      scfg->adaptive, scfg->conf_threshold, x, committed, last_argmax, stable,
                      done_dev, st));
  return DG_OK;
}

int dg_op_kv_append(const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_pool,
                    uint16_t *v_pool, const int32_t *page_table, int32_t n_layers,
                    int32_t n_pages, int32_t pos0, int32_t n_new, int32_t n_kv_heads,
                    int32_t head_dim, int32_t page_size, void *stream) {
  if (!k_new || !v_new || !k_pool || !v_pool || !page_table || head_dim % 8 || n_layers < 1 ||
      pos0 < 0 || n_new < 0 || pos0 + n_new > n_pages * page_size)
    return fail(DG_EINVAL, "bad arguments");
  CK(dg::kv_append((const bf16 *)k_new, (const bf16 *)v_new, (bf16 *)k_pool, (bf16 *)v_pool,
                   page_table, n_layers, n_pages, pos0, n_new, n_kv_heads, head_dim, page_size,
                   (cudaStream_t)stream));
  return DG_OK;
}

}  // extern "C"
