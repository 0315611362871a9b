// Host-side launchers shared between the translation units of libdg.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dg.h"
#include "common.cuh"

namespace dg {

// ---- misc kernels (kernels_misc.cu) ---------------------------------------
cudaError_t fill_weights(bf16 *dst, uint64_t n, uint64_t seed, uint32_t tid, uint64_t e0,
                         float std_dev, cudaStream_t st);
// A [rows][cols] weight matrix as operand tiles (tiled_index) whose rows
// [0, r1), [r1, r2), [r2, rows) are the generated tensors tid0, tid1, tid2.
cudaError_t fill_tiled_weights(bf16 *dst, int rows, int cols, int r1, int r2, uint32_t tid0, uint32_t tid1,
                               uint32_t tid2, uint64_t seed, float std_dev, cudaStream_t st);
cudaError_t fill_moe_weights(bf16 *wr, bf16 *wgu, bf16 *wd, int d, int E, int F, int layer,
                             uint64_t seed, float std_dev, cudaStream_t st);
cudaError_t fill_const(float *dst, size_t n, float v, cudaStream_t st);
cudaError_t rope_table(float *cos_t, float *sin_t, int max_pos, int head_dim, float base,
                       cudaStream_t st);
// n_req canvases of C positions (request b: sample seed + b), arrays [n_req C].
cudaError_t canvas_init(int *x, uint8_t *committed, int *last, int *stable, int C, int V,
                        uint64_t seed, int canvas, cudaStream_t st, int n_req = 1);
cudaError_t embed_rows(float *h, const bf16 *table, const int *ids, int T, int d, cudaStream_t st);
// out = RMSNorm(h) * gain (bf16), row-major, or as operand tiles (tiled_index)
// when `tiled`; out_lo (optional) the bf16 rounding of the remainder, same layout.
cudaError_t rmsnorm_rows(bf16 *out, const float *h, const float *gain, int T, int d, float eps,
                         cudaStream_t st, bf16 *out_lo = nullptr, bool tiled = false);
// Routing of one MoE layer (kernels_route.cu), two launches.
// moe_route: top-k of the router logits r = xn W_r^T (value desc, expert id
// asc; softmax gates over the selected logits) into ids / gates [T][k]; for
// every pair t*k+s its rank among the pairs of its token group (kRouteTok
// tokens) with the same expert into rank[T*k]; the group's pairs per expert
// into gcount[moe_group_count_ints(T, E)].  moe_norm_route first forms
// xn = RMSNorm(h) * gain (fp32 h [T][d]) and writes it.  d: a multiple of 64;
// E <= 256; k <= 16.
// moe_scatter: from those, the stable counting sort of the pairs by expert:
// offs[E+1], slot_row[T*k] (sorted row of pair t*k+s; pass the rank array in
// as slot_row, it is overwritten), the item tiles x_tiles (below), and
// work[2*max_work] = (expert, first row) items of up to `tile_rows` = 128 rows,
// *n_work.  `work` holds moe_work_ints() ints: the item list, then one
// counter per item and a unit counter used by moe_ffn, all zeroed here.
// max_work: the item capacity the work buffer was sized for (moe_max_work of
// the largest T it serves); moe_ffn must be given the same value.
// stats (optional, device, 2 x u64): += experts with at least one row, += T*k.
// Item tiles: item i's rows as d/64 operand tiles of 128 rows x 64 columns
// (16 KB each, item-major, row r's 16-byte chunk c at position c ^ (r % 8)),
// moe_item_tile_elems(max_work, d) elements in all.
constexpr int kRouteTok = 32;
inline size_t moe_item_tile_elems(int max_work, int cols) { return (size_t)max_work * 128 * cols; }
size_t moe_group_count_ints(int T, int E);
cudaError_t moe_norm_route(const float *h, const float *gain, float eps, bf16 *xn, const bf16 *wr, int T, int d,
                           int E, int k, int *ids, float *gates, int *rank, int *gcount, int *err,
                           cudaStream_t st);
cudaError_t moe_route(const bf16 *xn, const bf16 *wr, int T, int d, int E, int k, int *ids, float *gates,
                      int *rank, int *gcount, int *err, cudaStream_t st);
// A grid-wide barrier's words: the arrival count at [0] and the generation
// at [32], on its own 128-byte line (the arrivals' atomics do not share a
// line with the CTAs polling the generation).  Zeroed before first use.
constexpr int kGridBarInts = 64;

struct Fp8Experts;
cudaError_t moe_scatter(const bf16 *xn, const int *ids, const int *gcount, int *slot_row, int T, int d, int E,
                        int k, int tile_rows, bf16 *x_tiles, int *offs, int *work, int *n_work, int max_work,
                        cudaStream_t st, unsigned long long *stats = nullptr, const Fp8Experts *fp8 = nullptr);
// moe_norm_route (h != null) or moe_route, then moe_scatter, as one launch
// when the routing grid fits the machine (the scatter then runs in the
// routing kernel after a grid-wide barrier on bar, kGridBarInts zeroed ints), else as
// two; *launches (optional) receives 1 or 2.  slot_row serves as the rank
// array in between.
cudaError_t moe_route_scatter(const float *h, const float *gain, float eps, bf16 *xn, const bf16 *wr, int T, int d,
                              int E, int k, int *ids, float *gates, int *slot_row, int *gcount, bf16 *x_tiles,
                              int *offs, int *work, int *n_work, int max_work, int *bar, int *err, cudaStream_t st,
                              unsigned long long *stats = nullptr, int *launches = nullptr,
                              const Fp8Experts *fp8 = nullptr);
size_t moe_max_work(int T, int k, int E, int tile_rows);
// Gate/up units of one expert-FFN launch that may run split along K (the
// overflow past a whole number of waves); their part tickets follow the
// work list's counters.
constexpr int kFfnSplitUnits = 64;
// Work list, per-item counters, the unit counter and the part tickets.
size_t moe_work_ints(int T, int k, int E, int tile_rows);
// Partial-sum slots of split gate/up units for moe_ffn: one per SM, 128 KB each.
size_t moe_ffn_part_slots();
constexpr size_t kFfnPartSlotBytes = (size_t)2 * 128 * 128 * 4;
// Routed experts of one layer (kernels_moe.cu): act = SwiGLU(X Wg^T, X Wu^T),
// y = act Wd^T, for every work item of moe_scatter; one persistent launch.
// X: the item tiles of moe_scatter; wgu / wd: expert weights as operand tiles
// (the fill kernels' layout); act_tiles: moe_item_tile_elems(max_work, F)
// elements of scratch; y: [rows][d] bf16, row = sorted pair row.  part_buf
// (optional, part_slots slots of kFfnPartSlotBytes): when a launch's gate/up
// units exceed a whole number of waves by a few (at most a quarter of the
// SMs), those units run split along K, each part's sums summed in part order
// by the last part (bf16 experts only).
// The e4m3 expert path (kernels_moe.cu): gate/up weights as e4m3 operand
// tiles (the bytes of bf16 tiles [E][2][F][d/2]) with their rows' scale
// exponents kw [E][2][F]; the scatter writes the token rows as e4m3 tiles and
// their exponents kx [rows].
struct Fp8Experts {
  const uint8_t *wgu8;
  const int *kw;
  int *kx;
};
// Rows of n_mat bf16 operand-tile matrices [R][C] to e4m3 operand tiles and
// scale exponents [n_mat][R] (C a multiple of 128).
cudaError_t quantize_rows_e4m3(const bf16 *src, uint8_t *dst, int *exps, int n_mat, int R, int C,
                               cudaStream_t st);
cudaError_t moe_ffn(const bf16 *x_tiles, int rows, const bf16 *wgu, const bf16 *wd, const int *offs,
                    const int *work, const int *n_work, int max_work, int E, int d, int F, bf16 *act_tiles,
                    bf16 *y, int *err, cudaStream_t st, const Fp8Experts *fp8 = nullptr,
                    float *part_buf = nullptr, int part_slots = 0);
cudaError_t moe_combine(float *h, const bf16 *y, const float *gates, const int *slot_row, int T,
                        int k, int d, bool accumulate, cudaStream_t st);
// h[t] += sum_s gate * y (as moe_combine with accumulate), then the RMSNorm of
// the updated row with `gain` into x_tiles (bf16 operand tiles, tiled_index
// over [T][d]): the next layer's QKV input.  d <= 4096, a multiple of 64.
cudaError_t moe_combine_norm(float *h, const bf16 *y, const float *gates, const int *slot_row,
                             int T, int k, int d, const float *gain, float eps, bf16 *x_tiles,
                             cudaStream_t st);
cudaError_t kv_append(const bf16 *k_new, const bf16 *v_new, bf16 *k_pool, bf16 *v_pool,
                      const int *page_table, int L, int n_pages, int pos0, int n, int Hkv, int hd,
                      int pg, cudaStream_t st);

// ---- GEMM-based layer pieces (kernels_gemm.cu) -----------------------------
constexpr int kMaxRequests = 8;  // requests decoded together in one forward
// Rows of a forward that belong to several requests (multi-request batching):
// rows [b R, (b + 1) R) are request b's, its first at absolute position
// pos0[b] of that request, its K/V pages at page_table[b * pages_per_req ...].
// n_req = 1: one request, rows at pos0[0] + row.
struct RowSet {
  int n_req = 1, rows_per_req = 0, pages_per_req = 0;
  int pos0[kMaxRequests] = {};
  __host__ __device__ int req(int row) const { return n_req > 1 ? row / rows_per_req : 0; }
  __host__ __device__ int pos(int row) const {
    const int b = req(row);
    return pos0[b] + row - b * rows_per_req;
  }
};
struct QkvOut {
  bf16 *q;                // [T][Hq*hd]
  bf16 *k_pool, *v_pool;  // layer slice [n_pages][Hkv][pg][hd]
  const int *page_table;
  RowSet rows;            // positions and page-table slices of the rows
  int pg, Hq, Hkv, hd;
  const float *cos_t, *sin_t;  // [max_pos][hd/2]
};
// `err`: device error word set by a tensor-core GEMM whose bounded wait gave up.
// Operands are operand tiles (tiled_index): x_tiles / act_tiles [T][K],
// wqkv [(Hq + 2 Hkv) hd][d] (rows W_q, W_k, W_v), w [N][K].
// xchg: device scratch of gemm_xchg_bytes() for the split-K partial exchange
// (one buffer serves every call on a stream; calls must not overlap).
size_t gemm_xchg_bytes();
cudaError_t gemm_qkv(const bf16 *x_tiles, const bf16 *wqkv, int T, int d, const QkvOut &o, int *err,
                     float *xchg, cudaStream_t st);
cudaError_t gemm_residual(const bf16 *act_tiles, const bf16 *w, int T, int K, int N, float *h, int *err,
                          float *xchg, cudaStream_t st);  // h[T][N] += act[T][K] . w[N][K]^T
constexpr int kExpertTileRows = 128;  // token rows per expert work item (MMA N <= 128)
// xn_lo (optional): low part of a hi/lo split of the fp32 normalised rows;
// the logits are then w_out . (xn + xn_lo).
// dyn (optional, device): stream words taken from memory instead of seed/canvas/step.
// logits (optional, device [T][V] fp32): also written, from the same accumulators
// the partials are reduced from.
cudaError_t gemm_lm_head_partials(const bf16 *xn, const bf16 *xn_lo, const bf16 *w_out, int T, int d,
                                  int V, uint64_t seed, int canvas, int step, float inv_tau,
                                  void *partials, int *err, cudaStream_t st,
                                  const StepParams *dyn = nullptr, float *logits = nullptr,
                                  int rows_per_req = 0);
cudaError_t gemm_lm_head_logits(const bf16 *xn, const bf16 *xn_lo, const bf16 *w_out, int T, int d,
                                int V, float *logits, int *err, cudaStream_t st);

// A bounded wait that nothing completes (kernels_gemm.cu): gives up after
// limit_cycles and records code 99 in *err, as a kernel's timed-out wait does.
cudaError_t bounded_wait_selftest(int *err, long long limit_cycles, cudaStream_t st);

// ---- sampler (kernels_sampler.cu) -------------------------------------------
// out[i] = the sampler's Gumbel noise of Philox word words[i].
cudaError_t gumbel_noise(const uint32_t *words, float *out, size_t n, cudaStream_t st);
cudaError_t logits_partials(const float *logits, int rows, int V, uint64_t seed, int canvas,
                            int step, float inv_tau, void *partials, cudaStream_t st);
cudaError_t sampler_merge(const void *partials, int C, int V, int *argmax, float *conf,
                          int *gumbel, cudaStream_t st);
// Continuation of a device-side canvas loop: the rule kernel of a step inside
// a CUDA graph WHILE node sets the node's condition to "not done" (and to 0
// once `err` records a bounded wait that gave up) and, when the loop goes on,
// advances the step words in dyn to the next step (step + 1, its Gumbel
// counter word and its annealed 1 / temperature).
struct LoopCtl {
  int active;                         // 0: an ordinary step
  cudaGraphConditionalHandle handle;  // condition of the WHILE node
  float temp_start, temp_end;         // re-noise temperature schedule
  const int *err;                     // error word of the step's bounded waits
};
// Lockstep batching of n_req requests (canvases of C positions each, one rule
// block per request): req_done[b] this step's per-request decision, req_nk[b]
// the step at which request b's canvas finished (0: not yet; zeroed at canvas
// start), counter a zeroed int the blocks count themselves on.
struct BatchCtl {
  int n_req = 1;
  int *req_done = nullptr, *req_nk = nullptr, *counter = nullptr;
};
// dyn (optional, device): the step number is taken from dyn->step (and, in a
// loop, the next step's words are written back to it).  *done: the step's
// canvas (every request's canvas) is finished.
cudaError_t sampler_rule(const int *argmax, const float *conf, const int *gumbel, int C, int step,
                         int budget_N, int stable_steps, int adaptive, float conf_threshold,
                         int *x, uint8_t *committed, int *last, int *stable, int *done,
                         cudaStream_t st, StepParams *dyn = nullptr, LoopCtl loop = LoopCtl{},
                         BatchCtl bt = BatchCtl{});

// ---- attention (kernels_attn.cu) -------------------------------------------
struct AttnShape {
  int n_prefix, n_new, Hq, Hkv, hd, pg, causal;
  int n_pages = 0;  // physical pages of the pools when known (0: unknown)
  // several requests of n_new rows each (q and out hold n_req * n_new rows):
  // request b's keys start after req_prefix[b] cached ones, its pages at
  // page_table[b * pages_per_req ...]; n_req = 1: n_prefix, the whole table
  int n_req = 1, pages_per_req = 0;
  int req_prefix[kMaxRequests] = {};
};
// Device scratch the call needs (none: split-KV states merge on chip); ws and
// ws_bytes of attention() are accepted and unused.
size_t attention_workspace_bytes(const AttnShape &s);
int attention_launch_count(const AttnShape &s);
// err (optional, device, 2 ints): err[0] is set when a bounded wait of the kernel
// gives up, err[1] to 39 when a page index is outside the pools (its keys are skipped).
// out_tiles: out as operand tiles (tiled_index over [n_new][Hq hd]), else
// row-major [n_new][Hq][hd].
cudaError_t attention(const bf16 *q, const bf16 *k_pool, const bf16 *v_pool, const int *page_table,
                      const AttnShape &s, bf16 *out, void *ws, size_t ws_bytes, cudaStream_t st,
                      int *err = nullptr, bool out_tiles = false);

}  // namespace dg
