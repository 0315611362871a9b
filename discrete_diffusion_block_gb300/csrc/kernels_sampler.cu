// Commit / re-noise / adaptive-stop sampler of one denoising step.
//
// Reading of the rule (DiffusionGemma report §3.3 adaptive stopping; blog
// post "Once Written, a Prefix Becomes History": high-confidence positions
// lock in first while the rest keep being revised; report §4: multinomial
// re-noising): per position the argmax a and confidence conf = max softmax
// probability come from a full-vocabulary reduction; an uncommitted position
// commits to a when conf >= threshold or when a was unchanged for
// `stable_steps` consecutive steps, otherwise it is re-noised with a
// Gumbel-max sample g of its softmax; the canvas is done when every position
// is committed (adaptive) or at the budget N, where the rest take a.
//
// The reduction order is fixed so that results are reproducible bit for bit:
// 256-wide vocab tiles (row_tile_partial in sampler.cuh, the same code as the
// LM-head epilogue), merged by a balanced binary tree in tile order (left =
// lower vocab range).
#include "internal.h"
#include "sampler.cuh"

namespace dg {

namespace {

// One row of a vocabulary tile of fp32 logits in global memory.  A thread's
// chunk of 32 logits is one 128-byte line, read as eight 16-byte loads.
struct GlobalRowSrc {
  const float *row;  // the tile's 256 logits
  __device__ __forceinline__ void issue(int c, uint32_t *x) {
    const uint4 *p = reinterpret_cast<const uint4 *>(row + 32 * c);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 q = __ldg(p + j);
      x[4 * j] = q.x;
      x[4 * j + 1] = q.y;
      x[4 * j + 2] = q.z;
      x[4 * j + 3] = q.w;
    }
  }
  __device__ __forceinline__ void wait(uint32_t *) {}
};

constexpr int kPartialThreads = 256;

// One thread per (row, vocabulary tile), tiles of a row on consecutive
// threads; the reduction is row_tile_partial, the LM-head epilogue's code.
__global__ void __launch_bounds__(kPartialThreads) logits_partials_kernel(const float *logits, int rows,
                                                                          int V, uint32_t key0,
                                                                          uint32_t key1, uint32_t ctr2,
                                                                          float inv_tau, PartialPlanes P) {
  __shared__ float gbound[256];
  for (int b = threadIdx.x; b < 256; b += blockDim.x) gbound[b] = gumbel_bucket_bound(b);
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  const int tiles = V / kVocabTile;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)rows * tiles) return;
  const int r = (int)(idx / tiles), v = (int)(idx - (long long)r * tiles);
  GlobalRowSrc src{logits + (size_t)r * V + (size_t)v * kVocabTile};
  const Partial p = row_tile_partial(src, v, (uint32_t)r, ctr2, key0, key1, gbound, inv_tau);
  const size_t o = (size_t)r * tiles + v;
  P.m[o] = p.m;
  P.a[o] = p.a;
  P.s[o] = p.s;
  P.gk[o] = p.gk;
  P.gi[o] = p.gi;
}

__global__ void gumbel_noise_kernel(const uint32_t *words, float *out, size_t n) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    out[i] = gumbel(open_uniform(words[i]));
}

// Balanced binary tree over the tiles of one position; one block per position.
constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(PartialPlanes P, int tiles,
                                                              int leaves_per_thread, int *argmax,
                                                              float *conf, int *gumbel) {
  pdl_wait();
  pdl_trigger();
  const int pos = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // in-thread subtree over leaves [tid*c, tid*c + c), c a power of two
  Partial stack[12];
  int level[12];
  int sp = 0;
  for (int i = 0; i < leaves_per_thread; ++i) {
    const int t = tid * leaves_per_thread + i;
    Partial p = (t < tiles) ? P.load((size_t)pos * tiles + t) : empty_partial();
    int l = 0;
    while (sp > 0 && level[sp - 1] == l) {
      p = merge_partials(stack[sp - 1], p);
      --sp;
      ++l;
    }
    stack[sp] = p;
    level[sp] = l;
    ++sp;
  }
  Partial p = stack[0];
  // across the lanes of a warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    Partial o;
    o.m = __shfl_down_sync(0xffffffffu, p.m, off);
    o.a = __shfl_down_sync(0xffffffffu, p.a, off);
    o.s = __shfl_down_sync(0xffffffffu, p.s, off);
    o.gk = __shfl_down_sync(0xffffffffu, p.gk, off);
    o.gi = __shfl_down_sync(0xffffffffu, p.gi, off);
    if ((lane & (2 * off - 1)) == 0) p = merge_partials(p, o);
  }
  __shared__ Partial wres[kMergeThreads / 32];
  if (lane == 0) wres[warp] = p;
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < kMergeThreads / 32; w <<= 1)
      for (int i = 0; i + w < kMergeThreads / 32; i += 2 * w) wres[i] = merge_partials(wres[i], wres[i + w]);
    argmax[pos] = wres[0].a;
    conf[pos] = __fdiv_rn(1.0f, wres[0].s);
    gumbel[pos] = wres[0].gi;
  }
}

// One block per request (positions [b C, b C + C)).  With several requests
// (lockstep batching) a request whose canvas is finished (req_nk[b] > 0)
// keeps its state; req_nk[b] records the step at which its canvas finished,
// and the step is done when every request's canvas is; the last block to
// finish (a counter in global memory, fenced) takes that decision, continues
// a device loop and resets the counter.
__global__ void rule_kernel(const int *argmax, const float *conf, const int *gum, int C, int step,
                            int budget_N, int stable_steps, int adaptive, float thr, int *x,
                            uint8_t *committed, int *last, int *stable, int *done,
                            StepParams *dyn, LoopCtl loop, BatchCtl bt) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, i = b * C + threadIdx.x;
  if (dyn) step = dyn->step;
  const bool finished = bt.req_nk && bt.req_nk[b] > 0;
  bool com = true;
  if (threadIdx.x < C && !finished) {
    com = committed[i] != 0;
    if (!com) {
      const int a = argmax[i];
      const int st = (a == last[i]) ? stable[i] + 1 : 0;
      stable[i] = st;
      last[i] = a;
      com = (conf[i] >= thr) || (st >= stable_steps);
      x[i] = com ? a : gum[i];
      if (!com && step >= budget_N) {
        x[i] = a;
        com = true;
      }
      committed[i] = com ? 1 : 0;
    }
  }
  const int n_free = __syncthreads_count(!com);
  if (threadIdx.x != 0) return;
  const int d_req = (finished || step >= budget_N || (adaptive && n_free == 0)) ? 1 : 0;
  int d = d_req;
  if (gridDim.x > 1) {
    bt.req_done[b] = d_req;
    if (d_req && !finished) bt.req_nk[b] = step;
    __threadfence();
    if (atomicAdd(bt.counter, 1) != (int)gridDim.x - 1) return;  // not the last block
    __threadfence();
    for (int r = 0; r < (int)gridDim.x; ++r) d &= *(volatile int *)(bt.req_done + r);
    *bt.counter = 0;
  }
  *done = d;
  if (loop.active) {
    const bool stop = d || (loop.err && *(volatile const int *)loop.err);
    if (!stop && dyn) {  // the next step's words (the same schedule as the host's, in double)
      const int nx = step + 1;
      double tau = loop.temp_start;
      if (budget_N > 1) tau += ((double)loop.temp_end - (double)loop.temp_start) * (nx - 1) / (budget_N - 1);
      dyn->step = nx;
      dyn->ctr2 = (dyn->ctr2 & 0xFFFF0000u) | (uint32_t)nx;
      dyn->inv_tau = (float)(1.0 / tau);
    }
    cudaGraphSetConditional(loop.handle, stop ? 0u : 1u);
  }
}

}  // namespace

cudaError_t logits_partials(const float *logits, int rows, int V, uint64_t seed, int canvas,
                            int step, float inv_tau, void *partials, cudaStream_t st) {
  const int tiles = V / kVocabTile;
  const PartialPlanes P = PartialPlanes::at(partials, rows, tiles);
  const long long n = (long long)rows * tiles;
  if (n <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((n + kPartialThreads - 1) / kPartialThreads);
  return launch_pdl(logits_partials_kernel, dim3(blocks), dim3(kPartialThreads), 0, st, logits, rows, V,
                    (uint32_t)seed, (uint32_t)(seed >> 32), gumbel_ctr2(canvas, step), inv_tau, P);
}

cudaError_t gumbel_noise(const uint32_t *words, float *out, size_t n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  size_t blocks = (n + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  gumbel_noise_kernel<<<(unsigned)blocks, 256, 0, st>>>(words, out, n);
  return cudaGetLastError();
}

cudaError_t sampler_merge(const void *partials, int C, int V, int *argmax, float *conf,
                          int *gumbel, cudaStream_t st) {
  const int tiles = V / kVocabTile;
  int width = kMergeThreads;
  while (width < tiles) width *= 2;
  const int c = width / kMergeThreads;
  if (c > 1024) return cudaErrorInvalidValue;  // stack depth of the in-thread tree
  const PartialPlanes P = PartialPlanes::at(const_cast<void *>(partials), C, tiles);
  return launch_pdl(merge_kernel, dim3(C), dim3(kMergeThreads), 0, st, P, tiles, c, argmax, conf, gumbel);
}

cudaError_t sampler_rule(const int *argmax, const float *conf, const int *gumbel, int C, int step,
                         int budget_N, int stable_steps, int adaptive, float conf_threshold,
                         int *x, uint8_t *committed, int *last, int *stable, int *done,
                         cudaStream_t st, StepParams *dyn, LoopCtl loop, BatchCtl bt) {
  if (C > 1024 || bt.n_req < 1 || (bt.n_req > 1 && (!bt.req_done || !bt.req_nk || !bt.counter)))
    return cudaErrorInvalidValue;
  const int threads = ((C + 31) / 32) * 32;
  return launch_pdl(rule_kernel, dim3(bt.n_req), dim3(threads), 0, st, argmax, conf, gumbel, C, step, budget_N,
                    stable_steps, adaptive, conf_threshold, x, committed, last, stable, done, dyn, loop, bt);
}

}  // namespace dg
