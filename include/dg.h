/*
 * dg.h -- C ABI of the GB300 (sm_103a) block text-diffusion decoding library.
 *
 * The library runs the hot path of a DiffusionGemma-style decoder on one GPU:
 * a canvas of C = 256 tokens is refined by repeated denoising forwards that
 * attend to a read-only, paged bf16 KV cache of the clean prefix and
 * bidirectionally within the canvas; a top-k mixture-of-experts FFN follows
 * attention in every layer; an LM head fused with a vocabulary-split softmax
 * reduction feeds a commit / re-noise / adaptive-stop sampler; one extra
 * forward per finished canvas appends its K/V to the cache.
 *
 * Sources for what each call computes:
 *   DiffusionGemma Technical Report  -- abstract and §1 (256-token canvases
 *     refined in parallel; causal attention for context encoding,
 *     bidirectional attention for diffusion); §2.1 (canvas x_t in V^C,
 *     fully corrupted start x_1 ~ Unif(V^C)); §3.3 (adaptive stopping under a
 *     budget N = 48); §3.4 Eq. 7-10 (metrics; one extra forward between
 *     canvases appends the clean tokens' K/V); §4 (encoder KV cache of the
 *     prompt and previous canvases; multinomial corruption); §6 (batch-1
 *     serving; MoE, sampling and attention dominate step time).
 *   Blog post on the release, "Once Written, a Prefix Becomes History" --
 *     finished canvases become read-only prefix; high-confidence positions
 *     lock in first while the rest keep being revised.
 *
 * Conventions for every call
 *   - Return 0 (DG_OK) on success or a negative DG_E* code; the message of
 *     the last failure on the calling thread is dg_last_error().
 *   - Pointers documented as "host" are caller-owned host memory, read or
 *     written only during the call.  Pointers documented as "device" are
 *     device memory of the current CUDA device; the library never frees them.
 *   - A model owns its device memory (weights, KV pool, scratch) from
 *     dg_init_model until dg_free_model.  A model is not thread-safe; all of
 *     its work is ordered on its CUDA stream.  Calls that return host data
 *     synchronise that stream before returning.
 *   - Integer tensors are int32, "bf16" tensors hold IEEE bfloat16 bit
 *     patterns (uint16), float tensors are IEEE fp32; all row-major.
 */
#ifndef DG_H
#define DG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DG_OK 0
#define DG_EINVAL (-1)      /* bad argument or unsupported shape               */
#define DG_ENOMEM (-2)      /* device allocation failed                        */
#define DG_ECUDA (-3)       /* a CUDA call or kernel launch failed             */
#define DG_ESTATE (-4)      /* call out of order (e.g. denoise before prefill) */
#define DG_ECAPACITY (-5)   /* KV pool or position range exhausted             */
#define DG_ETIMEOUT (-6)    /* a bounded device-side wait gave up              */

/* Model shape.  Supported: head_dim in {64, 128}; d_model, n_q_heads*head_dim,
 * d_ff multiples of 64; vocab a multiple of 256; n_experts <= 256;
 * top_k <= 16; n_q_heads a multiple of n_kv_heads. */
typedef struct dg_config {
    int32_t n_layers;
    int32_t d_model;
    int32_t n_q_heads;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t n_experts;
    int32_t top_k;
    int32_t d_ff;          /* expert SwiGLU width F                          */
    int32_t vocab;
    int32_t page_size;     /* tokens per KV page (a multiple of 64)          */
    int32_t max_context;   /* KV pool capacity in tokens (prompt + canvases), per request */
    int32_t max_requests;  /* requests decoded together (0 or 1: one; at most 8), see
                              dg_generate_batch                                */
    int32_t expert_fp8;    /* 1: the experts' gate/up products in FP8 e4m3 (blog
                              "Test Conditions Behind 1,456 Tokens per Second":
                              FP8 serving): each W_gate / W_up row and each
                              expert input row stored as e4m3(row * 2^-k), k the
                              smallest integer with max|row| <= 448 * 2^k
                              (round to nearest even, saturating); W_down and
                              the SwiGLU output stay bf16; d_model a multiple
                              of 128.  The e4m3 copy is made from the bf16
                              weights at init (seeded or borrowed).  0: bf16.  */
    float rope_base;       /* RoPE theta base (10000)                        */
    float rms_eps;         /* RMSNorm epsilon (1e-6)                         */
    float init_std;        /* std of the seeded random-init weights (0.02)   */
    uint64_t weight_seed;  /* seed of the Philox weight stream               */
} dg_config;

/* Sampler of one canvas.  Commit rule: an uncommitted position commits to its
 * argmax when conf >= conf_threshold or when its argmax was unchanged for
 * stable_steps consecutive steps; every other position is re-noised with a
 * Gumbel-max sample of its softmax at temperature tau_n; the canvas stops
 * when all positions are committed (adaptive != 0) or after budget_N steps.
 * Temperature annealing (report §5, the online teacher's sampler): tau_n
 * moves linearly from temp_start at step 1 to temp_end at step budget_N,
 * tau_n = temp_start + (temp_end - temp_start) (n - 1) / (budget_N - 1) in
 * double, and the Gumbel keys are fp32(l * fp32(1 / tau_n)) + G; 1.0 and 1.0
 * sample the model's own softmax.  argmax and conf always use tau = 1. */
typedef struct dg_sampler_config {
    int32_t canvas_len;      /* C (256 in the method; 1..1024 supported)       */
    int32_t budget_N;        /* denoising budget N (48)                        */
    int32_t stable_steps;    /* 2                                              */
    int32_t adaptive;        /* 1: stop early once all committed               */
    int32_t eos_id;          /* -1: no end-of-sequence token                   */
    int32_t commit_causal;   /* 1: causal mask inside the canvas in the KV-append forward */
    float conf_threshold;    /* 0.9                                             */
    float temp_start;        /* re-noise temperature at step 1 (1.0; > 0)      */
    float temp_end;          /* ... and at step budget_N (1.0; > 0)            */
    uint64_t sample_seed;    /* seed of the canvas-init and Gumbel streams     */
} dg_sampler_config;

/* Eq. 7-10 of the report over one dg_generate call. */
typedef struct dg_stats {
    int32_t K;               /* canvases generated                             */
    int32_t total_tokens;    /* Eq. 7                                          */
    int32_t total_steps;     /* Eq. 8                                          */
    int32_t n_forwards;      /* denoise forwards + KV-append forwards          */
    double effective_steps;  /* Eq. 9                                          */
    double tpf;              /* Eq. 10                                         */
    double prefill_seconds;  /* wall time of the prompt encoding               */
    double decode_seconds;   /* wall time of the canvases (prefill excluded)   */
    double steps_per_s;      /* total_steps / decode_seconds                   */
    double tokens_per_s;     /* total_tokens / decode_seconds                  */
    int32_t canvas_loop_syncs; /* device->host synchronisations of the denoising loops */
    int32_t *N_k;            /* host, caller-owned, >= K_max entries, or NULL  */
    int32_t *C_k;            /* host, caller-owned, >= K_max entries, or NULL  */
} dg_stats;

typedef struct dg_model dg_model;

/* Message of the last failed call on this thread ("" if none). */
const char *dg_last_error(void);

/* Create a model on the current CUDA device: the paged KV pool for
 * cfg->max_context tokens, all scratch, and the weights.  `weights` NULL:
 * the model allocates and owns seeded random-init bf16 weights
 * (Philox4x32-10, see dg_op_fill_weights).  Otherwise weights[] holds
 * 3 + 7 * n_layers device pointers the model borrows (never writes or frees;
 * they must stay valid until dg_free_model), in the order of the DG_W_*
 * enum below: weights[0..2] = EMBED, LM_HEAD, FINAL_NORM; then for layer L,
 * weights[3 + 7 L + j], j = 0..6 = WQKV, WO, ROUTER, W_GATE_UP, W_DOWN,
 * ATTN_NORM, MOE_NORM, each in the physical layout dg_get_weight documents
 * (bf16 except the fp32 norm gains; device addresses 16-byte aligned).
 * `cuda_stream` (a cudaStream_t) orders all of the model's work; NULL
 * creates a private non-blocking stream.  On success *out owns everything
 * but borrowed weights until dg_free_model.  DG_ENOMEM if a device
 * allocation fails (everything allocated so far is released).
 * Host-side fault injection, read here from the environment (nothing is
 * done to the GPU): DG_FAULT=alloc:n (or DG_FAULT_ALLOC=n) -- the model's
 * n-th device allocation fails with DG_ENOMEM; DG_FAULT=badcall:n -- its
 * n-th kernel launch fails with DG_ECUDA before it is made; DG_FAULT=kvfull --
 * every KV capacity check fails with DG_ECAPACITY. */
int dg_init_model(const dg_config *cfg, const dg_sampler_config *scfg,
                  const void *const *weights, void *cuda_stream, dg_model **out);
void dg_free_model(dg_model *m);

/* Encode prompt_ids[0..n) (host) with causal attention at positions 0..n-1
 * and write their K/V into the cache (report §1, context encoding).  Resets
 * any previous generation.  n may be 0.  DG_ECAPACITY if the prompt plus one
 * canvas does not fit max_context. */
int dg_prefill(dg_model *m, const int32_t *prompt_ids, int32_t n);

/* One denoising step of the current canvas (the first call after prefill or
 * commit initialises it to uniform random ids, report §2.1).  All canvas
 * positions attend to the whole prefix and the whole canvas; the sampler
 * commits / re-noises and decides whether the canvas is finished.
 * *done (host) receives 1 when the canvas is finished, else 0. */
int dg_denoise_step(dg_model *m, int32_t *done);

/* Denoise the current canvas until it is done (report §3.3: adaptive
 * stopping under the budget N), as a device-side loop: a CUDA graph whose
 * conditional WHILE node repeats the denoising step while the sampler's done
 * flag is 0, the step's sampler advancing the step number, Gumbel counter and
 * annealed temperature on the device; the host synchronises once, at the
 * end.  The first step of a model (which sets kernel attributes) and steps
 * with per-kernel profiling on (dg_profile(m, 1)) run one by one instead.
 * The results are those of calling dg_denoise_step until it reports done.
 * *n_steps (host, may be NULL) receives the steps taken by this call. */
int dg_denoise_canvas(dg_model *m, int32_t *n_steps);

/* Finish the current canvas: copy its ids to out_ids (host, canvas_len
 * entries, may be NULL), set *out_valid (host, may be NULL) to C_k (tokens
 * before the first EOS, report §3.4), then run the single extra forward that
 * encodes the canvas (causal inside the canvas unless commit_causal == 0)
 * and appends its K/V to the prefix.  DG_ESTATE if the canvas is not done. */
int dg_commit_canvas(dg_model *m, int32_t *out_ids, int32_t *out_valid);

/* The whole block-diffusion generation of the report (§3.3 adaptive
 * stopping under a budget N; §3.4 Eq. 7-10 and the single extra forward
 * between canvases; §1 causal context encoding; blog "Once Written, a Prefix
 * Becomes History": finished canvases become read-only prefix): prefill of
 * the prompt, then up to K_max canvases, each denoised until done and, but
 * for the last, committed with its KV-append forward; generation stops after
 * the canvas holding the first EOS.  out_ids (host, K_max * canvas_len
 * entries) receives the canvases; stats (may be NULL) receives Eq. 7-10 and
 * the timings.  Each canvas is denoised as in dg_denoise_canvas: one
 * device->host synchronisation per canvas (stats->canvas_loop_syncs). */
int dg_generate(dg_model *m, const int32_t *prompt, int32_t n_prompt, int32_t K_max,
                int32_t *out_ids, dg_stats *stats);

/* ---- helpers: state access for replay tests and benchmarking ------------ */

/* ---- multi-request batching (lockstep) ------------------------------------
 * A model created with cfg->max_requests = B > 1 holds B requests, each with
 * its own prompt, KV pages (max_context tokens each) and canvas, and runs
 * every denoising forward and every KV-append forward over all B canvases at
 * once (B * canvas_len rows through the projections, the expert FFN and the
 * LM head: the expert weights streamed per step serve B requests; blog, on
 * serving throughput under concurrency).  Requests advance in lockstep: a
 * canvas step runs until every request's canvas is finished, a request whose
 * canvas finished earlier keeps it unchanged, and all requests commit
 * together.  Request b samples with sample_seed + b; given that seed, its
 * tokens, step counts and Eq. 7-10 are those of a single-request model.
 * The single-request calls above (dg_prefill, dg_denoise_step,
 * dg_denoise_canvas, dg_commit_canvas, dg_generate, dg_rewind,
 * dg_write_canvas, dg_canvas_logits) return DG_EINVAL on such a model; the
 * state readers report request 0. */

/* Encode prompts[b][0 .. lens[b]) (host) of every request b < B into its own
 * KV pages, as dg_prefill does for one. */
int dg_prefill_batch(dg_model *m, const int32_t *const *prompts, const int32_t *lens);

/* Denoise the current canvases until every request's is finished, as
 * dg_denoise_canvas (one device-side loop, one host synchronisation);
 * n_steps (host, B entries, may be NULL) receives, per request, the step at
 * which its canvas finished. */
int dg_denoise_canvas_batch(dg_model *m, int32_t *n_steps);

/* Finish the current canvases: ids to out_ids (host, B * canvas_len, may be
 * NULL), each request's C_k to out_valid (host, B, may be NULL), then one
 * KV-append forward of all B canvases (each after its own prefix). */
int dg_commit_canvas_batch(dg_model *m, int32_t *out_ids, int32_t *out_valid);

/* dg_generate for B requests in lockstep: out_ids (host, B * K_max *
 * canvas_len; request b's canvas k at (b K_max + k) canvas_len) and stats
 * (host, B entries, may be NULL; per request, its own N_k / C_k arrays).
 * A request's generation ends with its canvas holding the first EOS (its
 * later canvases are computed with the others and not reported); the batch
 * ends when every request has ended or after K_max canvases. */
int dg_generate_batch(dg_model *m, const int32_t *const *prompts, const int32_t *lens, int32_t K_max,
                      int32_t *out_ids, dg_stats *stats);

/* Replace the sampler configuration (e.g. a new sample_seed). */
int dg_set_sampler(dg_model *m, const dg_sampler_config *scfg);

/* Forget everything after the first n_prefix cached tokens (the prompt plus
 * whole committed canvases) and drop the current canvas.  The cached K/V of
 * those tokens are kept, so decoding can restart without a prefill. */
int dg_rewind(dg_model *m, int32_t n_prefix);

/* Current canvas and sampler state (host outputs, canvas_len entries each;
 * any pointer may be NULL).  *step = steps taken on this canvas,
 * *canvas_index = k (0-based), *prefix_len = cached tokens. */
int dg_read_canvas(dg_model *m, int32_t *ids, uint8_t *committed, int32_t *last_argmax,
                   int32_t *stable, int32_t *step, int32_t *canvas_index, int32_t *prefix_len);

/* Overwrite the current canvas state (host inputs, canvas_len entries) and its
 * step counter / canvas index; used to replay a step from recorded state. */
int dg_write_canvas(dg_model *m, const int32_t *ids, const uint8_t *committed,
                    const int32_t *last_argmax, const int32_t *stable, int32_t step,
                    int32_t canvas_index);

/* Per-position outputs of the last denoising step (host, canvas_len each):
 * argmax a_i, confidence conf_i = max softmax prob, Gumbel-max sample g_i. */
int dg_read_step_outputs(dg_model *m, int32_t *argmax, float *conf, int32_t *gumbel);

/* Run the denoising forward of the current canvas without sampling and write
 * its fp32 logits [canvas_len][vocab] to logits_dev (device).  Test hook. */
int dg_canvas_logits(dg_model *m, float *logits_dev);

/* Cached K/V of `layer` at positions pos0..pos0+n-1, read through the page
 * table into k_out/v_out (host, bf16 bits, [n][n_kv_heads][head_dim]). */
int dg_read_kv(dg_model *m, int32_t layer, int32_t pos0, int32_t n, uint16_t *k_out,
               uint16_t *v_out);

/* Expert choice of the last forward that ran `layer`'s MoE: ids (host,
 * [rows][top_k], up to max_rows rows, descending router logit), *n_rows =
 * tokens of that forward.  Lets a replay follow the GPU's top-k decision
 * where router logits are tied within rounding. */
int dg_read_routing(dg_model *m, int32_t layer, int32_t *ids, int32_t max_rows, int32_t *n_rows);

/* Expert input of the last MoE layer the last forward ran (the MoE RMSNorm's
 * bf16 output rows, which the router and the experts read): rows (host,
 * [rows][d_model] bf16 bits, up to max_rows rows), *n_rows = its rows,
 * *layer = that layer.  After a prefill chunk that is the second-to-last
 * layer (the last layer's MoE does not run: its output feeds no cached key);
 * after a canvas forward there are none (*n_rows = 0: the final norm has
 * replaced them).
 * Lets a replay take the FP8 path's per-row quantization decisions on the
 * same bf16 values as the kernels. */
int dg_read_moe_input(dg_model *m, uint16_t *rows, int32_t max_rows, int32_t *n_rows, int32_t *layer);

/* Page table (logical page -> physical page), host out, up to max_entries;
 * *n_pages = pages covering the prefix plus the current canvas. */
int dg_read_page_table(dg_model *m, int32_t *table, int32_t max_entries, int32_t *n_pages);

/* Device pointer and size of a weight tensor.  which: DG_W_* below; layer is
 * ignored for the embedding, LM head and final norm.  Physical layouts:
 *   EMBED            [V][d]
 *   LM_HEAD          operand tiles of [V][d]
 *   WQKV             operand tiles of         rows: W_q, then W_k, then W_v
 *                    [(Hq + 2 Hkv) * hd][d]
 *   WO               operand tiles of [d][Hq * hd]
 *   ROUTER           128-expert blocks of     block b: experts 128 b .. (rows =
 *                    [d/64] tiles             min(128, E - 128 b)); tile (b, j):
 *                                             those rows, columns 64 j .. 64 j + 63
 *   W_GATE_UP        per expert e: operand    W_gate,e first, then W_up,e
 *                    tiles of [F][d], twice
 *   W_DOWN           [E][d/128][F/64] tiles   tile (e, b, j): rows 128 b ..
 *                                             128 b + 127 of W_down,e; columns
 *                                             64 j .. 64 j + 63
 *   Operand tiles of a [rows][cols] matrix: 128-row blocks (the last one
 *   rows % 128 when that is not 0), each cols / 64 tiles of (block rows) x 64
 *   bf16 columns, contiguous per tile and row-major with 128-byte rows
 *   in which the 16-byte chunk c of row r sits at chunk position c ^ (r % 8)
 *   (the tensor core's 128-byte-swizzled operand order, so that one bulk
 *   copy stages a tile).
 *   ATTN_NORM, MOE_NORM, FINAL_NORM  [d] (fp32 gains, initialised to 1) */
enum {
    DG_W_EMBED = 0, DG_W_LM_HEAD = 1, DG_W_FINAL_NORM = 2, DG_W_WQKV = 3, DG_W_WO = 4,
    DG_W_ROUTER = 5, DG_W_GATE_UP = 6, DG_W_DOWN = 7, DG_W_ATTN_NORM = 8, DG_W_MOE_NORM = 9
};
int dg_get_weight(dg_model *m, int32_t which, int32_t layer, void **dev_ptr, size_t *bytes);

/* ---- profiling --------------------------------------------------------- */

/* Kernel classes of the decoder, for per-class timing and launch counts.
 * DG_K_ROUTE covers the routing (the MoE RMSNorm, router logits, top-k and
 * gates, and each routed pair's rank among its token group's pairs of the
 * same expert) and the scatter (the stable sort of the routed pairs by
 * expert, the gather of their rows into the expert FFN's operand tiles, and
 * its work list): one launch per MoE layer when the routing kernel's grid
 * fits the machine (the scatter then runs in its tail, after a grid-wide
 * barrier), else two. */
enum {
    DG_K_EMBED = 0, DG_K_RMSNORM, DG_K_QKV_ROPE, DG_K_ATTENTION, DG_K_O_PROJ,
    DG_K_ROUTE, DG_K_EXPERT_FFN, DG_K_COMBINE, DG_K_LM_HEAD,
    DG_K_SAMPLER_MERGE, DG_K_SAMPLER_RULE, DG_K_CANVAS_INIT, DG_K_CLASSES
};
const char *dg_kernel_class_name(int32_t cls);

/* Kernel launches are always counted per class.  enable = 1: every launch is
 * also bracketed by CUDA events on the model's stream (event-record nodes
 * inside captured steps) and the elapsed device time is accumulated per
 * class (read back at each synchronising call); enable = 2: counting only;
 * enable = 0: stop timing.  1 and 2 reset all counts, times and the expert
 * counters of dg_profile_experts. */
int dg_profile(dg_model *m, int32_t enable);
/* ms[DG_K_CLASSES] (host, may be NULL): accumulated device milliseconds;
 * launches[DG_K_CLASSES] (host, may be NULL): kernels launched per class. */
int dg_profile_read(dg_model *m, double *ms, int64_t *launches);

/* Since the last dg_profile(m, 1): sum over MoE launches of the experts that
 * received at least one row (each such expert's weights are streamed once
 * by the expert GEMMs) and of the routed (token, slot) rows.  Host outputs,
 * may be NULL. */
int dg_profile_experts(dg_model *m, int64_t *experts_touched, int64_t *rows_routed);

/* ---- kernel-level entry points (device pointers, caller's stream) ------- */

/* Seeded synthetic weights: dst[j] (device, bf16) = element e0 + j of tensor
 * `tensor_id`: an Irwin-Hall(4) sum of the four words of Philox4x32-10
 * (Salmon et al., SC'11) at counter (e mod 2^32, e div 2^32, tensor_id, 1),
 * key (seed mod 2^32, seed div 2^32):  s = sum_j (word_j >> 9),
 * w = fp32(s - 2^24) * fp32(std*sqrt(3)/2^23), rounded to bf16 (nearest even).
 * Tensor ids: 1 embedding, 2 LM head, 100 + 16*layer + {0 W_q, 1 W_k, 2 W_v,
 * 3 W_o, 4 router, 5 W_gate, 6 W_up, 7 W_down} (logical row-major shapes as
 * listed for dg_get_weight, expert tensors [E][F][d] / [E][d][F]). */
int dg_op_fill_weights(uint16_t *dst, uint64_t n, uint64_t seed, uint32_t tensor_id,
                       uint64_t e0, float std_dev, void *stream);

/* Status of the kernel-level entry points (dg_op_*) on the current device.
 * They are asynchronous on the caller's stream, so a failure inside a kernel
 * cannot be returned by the call that launched it: a bounded device-side wait
 * that gives up (about a second; the kernel then skips its remaining work and
 * its outputs are not valid), or an attention page-table entry outside the
 * pools, is recorded in a per-device status word that this call reads.  It
 * synchronises `stream`, returns DG_ETIMEOUT (a wait gave up), DG_ECUDA (a
 * kernel found itself launched without the thread-block cluster shape it
 * exchanges partial results in, and returned before touching anything) or
 * DG_EINVAL (a bad page index) when a kernel-level call since the last
 * dg_op_status recorded one, and clears the record; DG_OK otherwise.  The record is
 * shared by every kernel-level call on the device, and while it is set later
 * kernel-level kernels skip their waits (their outputs are not valid). */
int dg_op_status(void *stream);

/* Failure-detection self-test: launches one kernel that waits, with the
 * bounded wait every tensor-core kernel of the library uses, on an mbarrier
 * that nothing completes; after limit_cycles (1 .. 2^31 SM clock cycles) the
 * wait gives up and records code 99 in the status word, so that the next
 * dg_op_status on the stream returns DG_ETIMEOUT.  Nothing else is in flight
 * and the CUDA context stays usable.  No counterpart in the paper. */
int dg_op_wait_selftest(int64_t limit_cycles, void *stream);

/* Canvas attention (report §1, §4; blog "Once Written..."): for every query
 * position t < n_new (absolute position n_prefix + t) and query head h,
 *   out[t][h] = softmax_j(q[t][h] . k_j / sqrt(hd)) v_j
 * over keys j = 0 .. n_prefix + n_new - 1 of KV head h / (Hq/Hkv), where
 * causal == 0 lets every query see all keys (denoising) and causal != 0 hides
 * keys j > n_prefix + t (context encoding / KV append).
 *   q        device bf16 [n_new][Hq][hd] (already rotated)
 *   k_pool,
 *   v_pool   device bf16 pools of (page, KV head) blocks, [n_pages][Hkv] blocks
 *            of page_size * hd elements; key j lives in physical page
 *            page_table[j / page_size], slot s = j % page_size.  A block is
 *            hd/64 sub-blocks [page_size][64]: element f of slot s sits in
 *            sub-block f / 64, row s, at position 8 (((f % 64) / 8) ^ (s % 8))
 *            + f % 8 (the tensor core's 128-byte-swizzled operand order).  Keys are
 *            read in 64-key groups: the slots after the last key in its
 *            group (same page) are read too, weighted by zero, and must hold
 *            finite values (e.g. a zero-initialised pool)
 *   page_table device int32, >= ceil((n_prefix + n_new) / page_size) entries,
 *            each in [0, n_pages); an entry outside that range is not read
 *            (its keys are skipped) and is reported by dg_op_status
 *   n_pages  physical pages in each pool (>= 1, and n_pages * page_size >=
 *            n_prefix + n_new)
 *   out      device bf16 [n_new][Hq][hd]
 * workspace: device scratch of dg_op_attention_workspace_bytes() bytes.  The
 * split-KV partial softmax states are merged on chip (the blocks of a query
 * tile exchange them through distributed shared memory), so this is 0 for
 * every shape; the argument stays for callers that size it.  Timeouts and bad
 * page indices are reported by dg_op_status. */
size_t dg_op_attention_workspace_bytes(int32_t n_prefix, int32_t n_new, int32_t n_q_heads,
                                       int32_t n_kv_heads, int32_t head_dim);
int dg_op_canvas_attention(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                           const int32_t *page_table, int32_t n_prefix, int32_t n_new,
                           int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                           int32_t page_size, int32_t n_pages, int32_t causal, uint16_t *out,
                           void *workspace, size_t workspace_bytes, void *stream);

/* The canvas attention for callers that cannot allocate device memory or
 * hand the library a workspace: code whose device memory is owned and
 * budgeted entirely by a host framework (a serving engine's memory pool), a
 * plugin interface whose signature has no workspace argument, or a
 * latency-critical loop in which an allocation (which may synchronise the
 * device) is not acceptable.  The paper has no counterpart; this is a
 * property of the library, not of the method.
 *
 * Inputs, outputs and results as dg_op_canvas_attention.  The kernel needs no
 * device scratch (the split-KV partial states are merged in distributed
 * shared memory); the only device memory it touches besides its inputs and
 * outputs is the library's status word (see dg_op_status), a file-scope
 * device array of 256 bytes that every device loading the library holds
 * until exit.  Nothing is allocated or freed by this call.  The first
 * kernel-level call on a device looks up that array's device address (a
 * host-side query, once per device), so make it before any stream capture.
 * Calls that overlap on the GPU share the status word: a timeout recorded by
 * one is reported to whichever reads it first. */
int dg_op_canvas_attention_noalloc(const uint16_t *q, const uint16_t *k_pool,
                                   const uint16_t *v_pool, const int32_t *page_table,
                                   int32_t n_prefix, int32_t n_new, int32_t n_q_heads,
                                   int32_t n_kv_heads, int32_t head_dim, int32_t page_size,
                                   int32_t n_pages, int32_t causal, uint16_t *out, void *stream);

/* Mixture-of-experts FFN (report §6 "MoE"): for each of T rows of xn
 * (device bf16 [T][d], already RMS-normalised),
 *   r = xn W_r^T; S = the top_k largest r (ties -> lower expert id);
 *   gates = softmax(r_S); y = sum_{e in S} gate_e W_down,e (silu(W_gate,e xn) * W_up,e xn)
 * Weights in the layouts of dg_get_weight (W_GATE_UP, W_DOWN).  The SwiGLU
 * activations and each expert's output row are rounded to bf16 (the bf16
 * operands of the next product, and of the gate-weighted sum, which
 * accumulates in fp32).
 * Outputs (device): y fp32 [T][d]; expert_ids int32 [T][top_k] (descending
 * router logit); gates fp32 [T][top_k].  workspace: dg_op_moe_workspace_bytes(). */
size_t dg_op_moe_workspace_bytes(int32_t T, int32_t d, int32_t n_experts, int32_t top_k,
                                 int32_t d_ff);
int dg_op_moe(const uint16_t *xn, const uint16_t *w_router, const uint16_t *w_gate_up,
              const uint16_t *w_down, int32_t T, int32_t d, int32_t n_experts, int32_t top_k,
              int32_t d_ff, float *y, int32_t *expert_ids, float *gates, void *workspace,
              size_t workspace_bytes, void *stream);

/* Fill the three MoE weight tensors of `layer` (layouts of dg_get_weight) with
 * the seeded weights of tensor ids 100 + 16*layer + {4, 5, 6, 7}. */
int dg_op_fill_moe_weights(uint16_t *w_router, uint16_t *w_gate_up, uint16_t *w_down, int32_t d,
                           int32_t n_experts, int32_t d_ff, int32_t layer, uint64_t seed,
                           float std_dev, void *stream);

/* Per-(position, vocab tile) sampler partials (report §6 "GPU time
 * breakdown": sampling is one of the three dominant operations; the blog's
 * commit rule needs a full-vocabulary softmax per position).  Tiles are 256
 * vocab entries; inside tile t, in ascending v: m = max logit, a = first
 * index reaching it, s = left-to-right fp32 sum of dg_exp(l_v - m), (gk, gi)
 * = max and first argmax of fp32(l_v * inv_tau) + G_v (inv_tau = 1 / temperature
 * of the re-noise sample, 1.0 for the model's own softmax; see
 * dg_sampler_config) with Gumbel noise G_v = -dg_log(-dg_log(u))
 * and u = (2 (w >> 9) + 1) 2^-24, w = word (v mod 4) of Philox4x32-10 at
 * counter (v div 4, position, (canvas << 16) | step, 3), key = sample seed.
 * Layout of `partials` (device, rows * V/256 * 20 bytes): 5 planes of
 * [rows][V/256]: m (f32), a (i32), s (f32), gk (f32), gi (i32).
 * dg_op_lm_head_partials computes logits = (xn + xn_lo) W_out^T with fp32
 * accumulation in tensor memory and reduces them with the decoder's own
 * LM-head epilogue, the logits never leaving the chip.  xn and xn_lo (may be
 * NULL: the low half of a hi/lo split of fp32 rows, as the decoder's final
 * norm writes it) are device bf16 operand tiles of [rows][d], w_out device
 * bf16 operand tiles of [V][d] (layout of dg_get_weight; see
 * dg_op_fill_tiled_weights).  When `logits` (device fp32 [rows][V]) is not
 * NULL the same launch also writes the logits the partials were reduced from.
 * dg_op_logits_partials runs the same per-(row, tile) reduction code on
 * given fp32 logits [rows][V] (device): the injected-logit entry of the
 * sampler, bit-identical to the epilogue on the same logits. */
int dg_op_lm_head_partials(const uint16_t *xn, const uint16_t *xn_lo, const uint16_t *w_out,
                           int32_t rows, int32_t d, int32_t V, uint64_t sample_seed,
                           int32_t canvas, int32_t step, float inv_tau, void *partials,
                           float *logits, void *stream);
int dg_op_logits_partials(const float *logits, int32_t rows, int32_t V, uint64_t sample_seed,
                          int32_t canvas, int32_t step, float inv_tau, void *partials,
                          void *stream);

/* dst (device, bf16, rows * cols elements; cols a multiple of 64) = the
 * operand tiles (layout of dg_get_weight) of the logical [rows][cols] tensor
 * `tensor_id` of the seeded weights (elements as dg_op_fill_weights). */
int dg_op_fill_tiled_weights(uint16_t *dst, int32_t rows, int32_t cols, uint64_t seed,
                             uint32_t tensor_id, float std_dev, void *stream);

/* The sampler's Gumbel noise transform: out[i] = -dg_log(-dg_log(u)),
 * u = (2 (words[i] >> 9) + 1) 2^-24 (device uint32 in, device fp32 out, n
 * entries).  Test hook: lets the transform be compared with a reference over
 * every distinct input. */
int dg_op_gumbel_noise(const uint32_t *words, float *out, uint64_t n, void *stream);

/* The FP8 expert path's weight quantizer (dg_config.expert_fp8): n_mat bf16
 * matrices [rows][cols] in operand tiles (contiguous, rows * cols elements
 * each; cols a multiple of 128) to e4m3 (fn) operand tiles (rows * cols bytes
 * each: the bytes of bf16 tiles [rows][cols/2]; element (r, c) of a 128-row
 * block at k-tile c / 128, 16-element chunk ((c % 128) / 16) ^ (r % 8)) and
 * each row's scale exponent k (exps [n_mat][rows]): row = e4m3 row * 2^k, k
 * the smallest integer with max|row| <= 448 * 2^k (0 for a zero row),
 * conversion rounding to nearest even and saturating.  Device pointers; the
 * caller owns them.  No counterpart in the paper beyond "FP8 weights". */
int dg_op_quantize_rows_e4m3(const uint16_t *src, int32_t n_mat, int32_t rows, int32_t cols, uint8_t *dst,
                             int32_t *exps, void *stream);

/* Merge the partials of each row by a balanced binary tree over the tiles
 * (left = lower vocab range; M = max; S = sL*exp(mL-M) + sR*exp(mR-M);
 * argmax / Gumbel winner from the right only if strictly greater) and apply
 * the commit / re-noise / stop rule to the canvas state (all device, C
 * entries): x, committed (uint8), last_argmax, stable.  step is 1-based.
 * Outputs (device): argmax, conf (= 1/S), gumbel, and *done_dev (int32). */
int dg_op_sampler_update(const void *partials, int32_t C, int32_t V, int32_t step,
                         const dg_sampler_config *scfg, int32_t *x, uint8_t *committed,
                         int32_t *last_argmax, int32_t *stable, int32_t *argmax, float *conf,
                         int32_t *gumbel, int32_t *done_dev, void *stream);

/* KV append, standalone: copy n_layers x n_new tokens of K and V (device bf16
 * [n_layers][n_new][Hkv][hd]) into the pools (device bf16, n_layers pools in
 * the layout of dg_op_canvas_attention) at absolute positions
 * pos0 .. pos0+n_new-1 through page_table (device int32). */
int dg_op_kv_append(const uint16_t *k_new, const uint16_t *v_new, uint16_t *k_pool,
                    uint16_t *v_pool, const int32_t *page_table, int32_t n_layers,
                    int32_t n_pages, int32_t pos0, int32_t n_new, int32_t n_kv_heads,
                    int32_t head_dim, int32_t page_size, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* DG_H */
