// Routing of one MoE layer (report §6 "MoE"; DiffusionGemma model card,
// "Architecture": 128 experts, 8 active per token) in two launches.
//
// route_kernel: the layer's RMSNorm (optional), the router logits
// r = xn W_r^T, the top-k experts of every token with their softmax gates,
// and each routed (token, slot) pair's rank among the pairs of its token
// group that chose the same expert.  A CTA owns 32 tokens (the MMA N) and 1/S
// of the model dimension; the S CTAs of one token group form a cluster.
//   1. (norm) each CTA sums the squares of its slice of the 32 rows; the S
//      partial sums are exchanged through distributed shared memory and added
//      in rank order, so every CTA derives the same 1/rms.  It writes its
//      slice of xn (bf16) to global memory and, 128-byte swizzled, to shared
//      memory as the MMA B operand.  Without the norm, the B slice is loaded
//      from xn with TMA.
//   2. one thread streams the CTA's K-slice of W_r (stored as operand tiles,
//      one bulk copy per 128-expert x 64 tile; weights never change, so they
//      are requested before the wait on the previous kernel) and four
//      threads in four warps issue tcgen05.mma (M = 128 experts, N = 32
//      tokens), each into its own 32-column TMEM accumulator per 128 experts
//      over every fourth K step, so that short MMAs are issued in parallel.
//   3. the four accumulators are summed into the CTA's partial logits; CTA
//      z receives the partials of its 32/S tokens from every peer (bulk
//      shared-to-shared copies), adds the S partials in rank order
//      (deterministic), and one warp per token selects the top k.
//   4. per-CTA expert counts are exchanged in the cluster: each pair gets its
//      rank within the group, and the group's per-expert counts go to global
//      memory.
// scatter_kernel: every block turns the group counts into expert offsets
// (the stable counting sort's prefix sums: groups, then experts), places its
// share of the pairs at offs[e] + (pairs of e in earlier groups) + rank, and
// copies their token rows there; block 0 also writes the work list.  The
// result is the order of a stable sort of the pairs by expert.
// Every mbarrier wait is bounded (error word + abort flag); every CTA passes
// the same cluster barriers whatever happened, so no CTA can be left waiting.
#include <cuda.h>

#include <cstdlib>

#include "gemm_tc.cuh"
#include "internal.h"

namespace dg {

cudaError_t tmap_bf16_cached(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols,
                             uint32_t box);

namespace {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kTokThreads = kRouteThreads / kRouteTok;  // threads per token in the norm
constexpr uint32_t kWBox = 128 * 128;              // 128 experts x 64 bf16
constexpr uint32_t kXBox = kRouteTok * 128;        // 32 tokens x 64 bf16
constexpr int kNormRegs = 12;
constexpr int kPairIters = kRouteTok * 16 / kRouteThreads;  // pairs per thread at most (k <= 16)  // float4 columns per thread held in registers by the norm
constexpr int kSmemBudget = 200 * 1024;  // dynamic; the expert sort adds 11 KB of static shared memory

// ---------------------------------------------------------------------------
// Placement of the routed pairs and copy of their token rows.
// ---------------------------------------------------------------------------
constexpr int kScatThreads = 256;

__host__ __device__ inline size_t scatter_smem_ints(int ng, int E, int per) { return (size_t)ng * E + 2 * E + 2 * (size_t)per; }
// Bytes of the table above, rounded up to 16 (the staged rows follow it).
__host__ __device__ inline size_t scatter_tab_bytes(int ng, int E, int per) { return (scatter_smem_ints(ng, E, per) * 4 + 15) & ~(size_t)15; }
// Staging for n_tok token rows of width d: the bf16 rows, and with fp8 their
// e4m3 codes (16-byte aligned) and scale exponents.
__host__ __device__ inline size_t scatter_stage_bytes(int n_tok, int d, int fp8) {
  const size_t rows = (size_t)n_tok * d * 2;
  return fp8 ? rows + (((size_t)n_tok * d + 15) & ~(size_t)15) + (size_t)n_tok * 4 : rows;
}

struct ScatArgs {
  const bf16 *xn;
  const int *ids, *gcount;
  int *slot_row;  // in: rank within the token group; out: sorted row
  bf16 *x_tiles;  // [item][d/64] tiles of 128 rows x 64 columns, swizzled
  int T, d, E, k, tile_rows, ng;
  int per;        // pairs per block
  int stage_bytes;  // shared memory after the table for the block's token rows (0: none)
  int fp8;        // rows written as e4m3 operand tiles ([item][d/128], 16 KB each) with exponents kx
  int *kx;        // fp8: scale exponent of every sorted row
  int *offs, *work, *n_work, *sync;
  int max_work;
  unsigned long long *stats;
};

// Exclusive prefix sum over the block of one value per thread (kScatThreads
// threads); returns the prefix and stores the block total in *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_tot, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncwarp();
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kScatThreads / 32; ++w) {
    const int c = warp_tot[w];
    before += w < warp ? c : 0;
    all += c;
  }
  __syncwarp();
  __syncthreads();  // warp_tot may be reused by the next scan
  *total = all;
  return before + x - v;
}

// The token rows t_lo .. t_lo + n_tok - 1 of a block's pairs (contiguous in
// xn) into shared memory, every 16-byte load of a round in flight, read
// through L2 (peers of the block may have written them).
__device__ __forceinline__ void scatter_stage_rows(const ScatArgs &a, int t_lo, int n_tok, uint4 *st4) {
  const uint4 *src = (const uint4 *)(a.xn + (size_t)t_lo * a.d);
  const int n4 = n_tok * (a.d / 8);
  for (int i0 = 0; i0 < n4; i0 += 8 * kScatThreads) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + (int)threadIdx.x + u * kScatThreads;
      if (i < n4) v[u] = __ldcg(src + i);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + (int)threadIdx.x + u * kScatThreads;
      if (i < n4) st4[i] = v[u];
    }
  }
}

// The block's first token row and token count.
__device__ __forceinline__ void scatter_tokens(const ScatArgs &a, int blk, int *t_lo, int *n_tok) {
  const int p0 = blk * a.per, p1 = min(a.T * a.k, p0 + a.per);
  *t_lo = p0 / a.k;
  *n_tok = p1 > p0 ? (p1 - 1) / a.k - *t_lo + 1 : 0;
}

// The scatter work of block `blk` (kScatThreads threads): its share of the
// pairs, and (blk 0) the expert segments, the work list and the FFN's
// counters.  tab: shared memory of scatter_smem_ints() ints; stage: shared
// memory of stage_bytes bytes (16-byte aligned) for the block's token rows,
// or null.
__device__ __forceinline__ void scatter_block(const ScatArgs &a, int blk, int *tab, int *warp_tot,
                                              unsigned char *stage, size_t stage_bytes, bool rows_staged = false) {
  // [ng][E]: pairs of e in earlier groups; then offs[E], first item[E]; then
  // the expert and group rank of each of this block's pairs
  const int E = a.E, ng = a.ng, n = ng * E;
  int *soffs = tab + n, *stoff = soffs + E, *s_ex = stoff + E, *s_rk = s_ex + a.per;
  const int TK = a.T * a.k;
  const int p0 = blk * a.per, p1 = min(TK, p0 + a.per);
  // the block's pairs and the group counts: every load of a round in
  // flight before any store (each load waits an L2 round trip)
  constexpr int kLoadU = 8;
  for (int i0 = 0; i0 < max(p1 - p0, n); i0 += kLoadU * kScatThreads) {
    int ex[kLoadU], rk[kLoadU], gc[kLoadU];
#pragma unroll
    for (int u = 0; u < kLoadU; ++u) {
      const int i = i0 + (int)threadIdx.x + u * kScatThreads;
      if (i < p1 - p0) {
        ex[u] = a.ids[p0 + i];
        rk[u] = a.slot_row[p0 + i];
      }
      if (i < n) gc[u] = a.gcount[i];
    }
#pragma unroll
    for (int u = 0; u < kLoadU; ++u) {
      const int i = i0 + (int)threadIdx.x + u * kScatThreads;
      if (i < p1 - p0) {
        s_ex[i] = ex[u];
        s_rk[i] = rk[u];
      }
      if (i < n) tab[i] = gc[u];
    }
  }
  __syncwarp();
  __syncthreads();
  const int e = threadIdx.x;  // E <= kScatThreads
  int tot = 0;
  if (e < E)
    for (int g = 0; g < ng; ++g) {
      const int c = tab[g * E + e];
      tab[g * E + e] = tot;
      tot += c;
    }
  int total, n_items;
  const int off = block_exclusive_scan(tot, warp_tot, &total);
  const int tiles = e < E ? (tot + a.tile_rows - 1) / a.tile_rows : 0;
  const int toff = block_exclusive_scan(tiles, warp_tot, &n_items);
  if (e < E) {
    soffs[e] = off;
    stoff[e] = toff;
  }
  if (blk == 0) {  // the expert segments and the work list of the expert FFN
    int touched;
    block_exclusive_scan(e < E && tot > 0 ? 1 : 0, warp_tot, &touched);
    if (e < E) {
      a.offs[e] = off;
      for (int j = 0; j < tiles; ++j) {
        a.work[2 * (toff + j)] = e;
        a.work[2 * (toff + j) + 1] = j * a.tile_rows;
      }
    }
    if (threadIdx.x == 0) {
      a.offs[E] = total;
      *a.n_work = n_items;
      if (a.stats) {  // experts whose weights the expert FFN streams, and their rows
        atomicAdd(&a.stats[0], (unsigned long long)touched);
        atomicAdd(&a.stats[1], (unsigned long long)total);
      }
    }
    for (int i = threadIdx.x; i <= a.max_work + kFfnSplitUnits; i += kScatThreads) a.sync[i] = 0;  // FFN counters
  }
  __syncwarp();
  __syncthreads();
  // The block's pairs are consecutive, so their tokens are the few rows
  // t_lo .. t_hi (k pairs each): when they fit, those rows are staged in
  // shared memory once (every 16-byte load in flight together) and each pair
  // is written from there.
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, vec = a.d / 8, KT = a.d / 64;
  constexpr int NW = kScatThreads / 32;
  const int t_lo = p0 / a.k, n_tok = p1 > p0 ? (p1 - 1) / a.k - t_lo + 1 : 0;
  if (stage && scatter_stage_bytes(n_tok, a.d, a.fp8) <= stage_bytes) {
    uint4 *st4 = (uint4 *)stage;
    if (!rows_staged) {  // (the fused kernel may have staged them before its grid barrier)
      scatter_stage_rows(a, t_lo, n_tok, st4);
      __syncthreads();
    }
    if (a.fp8) {
      // Each token's row is quantized once (one warp per token): its scale
      // exponent from the row maximum, then its e4m3 codes, in column order,
      // into shared memory after the staged rows.  One warp per pair then
      // copies its token's codes into row r of its item's e4m3 tiles (128
      // elements a k-tile; chunk j at position j ^ (r % 8)).
      unsigned char *q8 = stage + (size_t)n_tok * a.d * 2;
      int *texp = (int *)(q8 + (((size_t)n_tok * a.d + 15) & ~(size_t)15));
      for (int tt = warp; tt < n_tok; tt += NW) {
        const uint4 *row = st4 + (size_t)tt * vec;
        float amax = 0.0f;
        for (int c = lane; c < vec; c += 32) {
          const uint4 v = row[c];
          const __nv_bfloat162 *p2 = (const __nv_bfloat162 *)&v;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(p2[i]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const int kexp = e4m3_scale_exp(amax);
        uint4 *dst = (uint4 *)(q8 + (size_t)tt * a.d);
        for (int j = lane; j < a.d / 16; j += 32) {
          uint4 v[2] = {row[2 * j], row[2 * j + 1]};
          const __nv_bfloat162 *p2 = (const __nv_bfloat162 *)v;
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 x0 = __bfloat1622float2(p2[2 * i]), x1 = __bfloat1622float2(p2[2 * i + 1]);
            w[i] = cvt_e4m3x2(ldexpf(x0.x, -kexp), ldexpf(x0.y, -kexp)) |
                   (cvt_e4m3x2(ldexpf(x1.x, -kexp), ldexpf(x1.y, -kexp)) << 16);
          }
          dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (lane == 0) texp[tt] = kexp;
      }
      __syncthreads();
      for (int p = p0 + warp; p < p1; p += NW) {
        const int ex = s_ex[p - p0], t = p / a.k, g = t / kRouteTok;
        const int within = tab[g * E + ex] + s_rk[p - p0];
        if (lane == 0) a.slot_row[p] = soffs[ex] + within;
        const int item = stoff[ex] + within / a.tile_rows, rr = within % a.tile_rows;
        const uint4 *src = (const uint4 *)(q8 + (size_t)(t - t_lo) * a.d);
        unsigned char *dst8 = (unsigned char *)a.x_tiles + (size_t)item * (a.d / 128) * 16384 + (size_t)rr * 128;
        for (int j = lane; j < a.d / 16; j += 32) {
          const int kt = j >> 3, ch = j & 7;
          *(uint4 *)(dst8 + (size_t)kt * 16384 + ((ch ^ (rr & 7)) << 4)) = src[j];
        }
        if (lane == 0) a.kx[soffs[ex] + within] = texp[t - t_lo];
      }
      return;
    }
    // One warp per pair: the token's row into row r of its item's tiles
    // (16-byte chunk c of k-tile kt at chunk position c ^ (r % 8): the tensor
    // core's swizzled operand order).
    for (int p = p0 + warp; p < p1; p += NW) {
      const int ex = s_ex[p - p0], t = p / a.k, g = t / kRouteTok;
      const int within = tab[g * E + ex] + s_rk[p - p0];  // rank among the expert's rows
      if (lane == 0) a.slot_row[p] = soffs[ex] + within;
      const int item = stoff[ex] + within / a.tile_rows, rr = within % a.tile_rows;
      const uint4 *row = st4 + (size_t)(t - t_lo) * vec;
      uint4 *dst = (uint4 *)(a.x_tiles + (size_t)item * KT * (128 * 64)) + rr * 8;
      for (int c = lane; c < vec; c += 32) dst[(c >> 3) * 1024 + ((c & 7) ^ (rr & 7))] = row[c];
    }
    return;
  }
  // Otherwise one warp per pair, two pairs at a time; the warp copies the
  // token's row into row r of its item's tiles (16-byte chunk c of
  // k-tile kt at chunk position c ^ (r % 8): the tensor core's swizzled
  // operand order), both rows' loads in flight before any store.
  constexpr int U = 12;
  for (int pb = p0 + warp; pb < p1; pb += 2 * NW) {
    const uint4 *src[2];
    uint4 *dst[2];
    int rr[2];
    bool ok[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int p = pb + q * NW;
      ok[q] = p < p1;
      src[q] = nullptr;
      dst[q] = nullptr;
      rr[q] = 0;
      if (ok[q]) {
        const int ex = s_ex[p - p0], t = p / a.k, g = t / kRouteTok;
        const int within = tab[g * E + ex] + s_rk[p - p0];  // rank among the expert's rows
        if (lane == 0) a.slot_row[p] = soffs[ex] + within;
        const int item = stoff[ex] + within / a.tile_rows;
        rr[q] = within % a.tile_rows;
        src[q] = (const uint4 *)(a.xn + (size_t)t * a.d);
        dst[q] = (uint4 *)(a.x_tiles + (size_t)item * KT * (128 * 64)) + rr[q] * 8;
      }
    }
    for (int c0 = 0; c0 < vec; c0 += 32 * U) {
      uint4 v[2][U];
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = c0 + lane + 32 * u;
          if (ok[q] && c < vec) v[q][u] = src[q][c];
        }
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = c0 + lane + 32 * u;
          if (ok[q] && c < vec) dst[q][(c >> 3) * 1024 + ((c & 7) ^ (rr[q] & 7))] = v[q][u];
        }
    }
  }
}

__global__ void __launch_bounds__(kScatThreads) scatter_kernel(ScatArgs a) {
  extern __shared__ int tab[];
  __shared__ int warp_tot[kScatThreads / 32];
  pdl_wait();
  pdl_trigger();
  scatter_block(a, blockIdx.x, tab, warp_tot,
                a.stage_bytes ? (unsigned char *)tab + scatter_tab_bytes(a.ng, a.E, a.per) : nullptr,
                (size_t)a.stage_bytes);
}

struct RouteArgs {
  const float *h;      // norm: input rows fp32 [T][d]
  const float *gain;   // norm: RMSNorm gain [d]
  const bf16 *wr;      // router weights as operand tiles (rows = experts, the last block partial)
  float eps;
  bf16 *xn;            // norm: normalised rows out [T][d]
  int T, d, E, k, tile_rows;
  int S, nk_max, stages, m_tiles;  // cluster size, k-tiles per CTA (max), ring depth, 128-expert tiles
  int *ids;
  float *gates;
  int *rank;           // [T*k] rank of each pair among its group's pairs of the same expert
  int *gcount;         // [ceil(T/32)][E] pairs per (token group, expert)
  int *err;
  // fused scatter: after a grid-wide barrier (bar: kGridBarInts words), every
  // CTA runs its share of the scatter (sc, with sc.per pairs per CTA)
  int fuse;
  int grid;  // fused: CTAs of the launch
  int *bar;
  ScatArgs sc;
};

struct RouteSmem {
  uint32_t w_off, x_off, part_off, recv_off, logit_off, ss_off, cnt_off, pid_off, bars_off, bytes;
};

__host__ __device__ inline RouteSmem route_smem(int S, int nk_max, int stages, int m_tiles) {
  RouteSmem s;
  const int ep = m_tiles * 128;
  s.w_off = 0;
  s.x_off = s.w_off + (uint32_t)stages * m_tiles * kWBox;
  s.part_off = s.x_off + (uint32_t)nk_max * kXBox;
  s.recv_off = s.part_off + (uint32_t)kRouteTok * ep * 4;           // [S][32/S tokens][ep] from the peers
  s.logit_off = s.recv_off + (uint32_t)kRouteTok * ep * 4;
  s.ss_off = s.logit_off + (uint32_t)(kRouteTok / S) * ep * 4;
  s.cnt_off = s.ss_off + kRouteTok * 4;
  s.pid_off = s.cnt_off + ep * 4;
  s.bars_off = (s.pid_off + (uint32_t)(kRouteTok / S) * 16 * 4 + 15) & ~15u;
  s.bytes = s.bars_off + (8 + 8 + 3) * 8 + 32 + 1024;  // full[8], empty[8], x, acc, recv; words; alignment slack
  return s;
}

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   tc::smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
               : "memory");
}

// K-tile kt of every 128-expert block of W_r into one ring stage: block m
// holds min(128, E - 128 m) rows, contiguous per k-tile.
__device__ __forceinline__ void load_w_tile(const bf16 *wr, int E, int KT, int m_tiles, int kt, unsigned char *stage,
                                            uint64_t *bar, bool expect = true) {
  if (expect) tc::mbar_expect_tx(bar, (uint32_t)E * 128);
  for (int mt = 0; mt < m_tiles; ++mt) {
    const int rows = min(128, E - 128 * mt);
    bulk_load(stage + mt * kWBox, wr + ((size_t)128 * KT * mt + (size_t)rows * kt) * 64, (uint32_t)rows * 128, bar);
  }
}

__device__ __forceinline__ int ld_acquire_s32(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Arrival with release at gpu scope: the writes this thread has observed
// (the CTA's, through the preceding CTA barrier) are visible before the count.
__device__ __forceinline__ int atom_add_release_s32(int *p, int v) {
  int old;
  asm volatile("atom.add.release.gpu.global.s32 %0, [%1], %2;\n" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void st_release_s32(int *p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(addr));
  return v;
}

// Order-preserving map of a float onto an unsigned key (larger float, larger
// key; -0 and +0 equal).  Key 0 is below every non-NaN value.
__device__ __forceinline__ unsigned float_key(float f) {
  unsigned u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(unsigned key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Top-k of one token's E <= 256 logits (shared memory) by one warp: value
// descending, lower expert id first among equal values; gates are the softmax
// of the selected logits.
__device__ __forceinline__ void topk_warp(const float *lrow, int E, int k, int lane, int *ids_out,
                                          float *gates_out, int *ids_smem) {
  unsigned key[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = lane + 32 * j;
    key[j] = e < E ? float_key(lrow[e]) : 0u;
  }
  float my_val = 0.0f;
  int my_id = 0;
  for (int s = 0; s < k; ++s) {
    unsigned bk = 0u, be = 0xffffffffu;
#pragma unroll
    for (int j = 0; j < 8; ++j)  // ascending expert id: strict > keeps the lowest id of a tie
      if (key[j] > bk) {
        bk = key[j];
        be = (unsigned)(lane + 32 * j);
      }
    const unsigned mk = __reduce_max_sync(0xffffffffu, bk);
    const unsigned me = __reduce_min_sync(0xffffffffu, bk == mk ? be : 0xffffffffu);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (me == (unsigned)(lane + 32 * j)) key[j] = 0u;  // taken
    if (lane == s) {
      my_val = key_float(mk);
      my_id = (int)me;
    }
  }
  const float top = __shfl_sync(0xffffffffu, my_val, 0);
  const float ex = lane < k ? expf(my_val - top) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    ids_out[lane] = my_id;
    ids_smem[lane] = my_id;
    gates_out[lane] = ex / sum;
  }
}

// ---- fused scatter ---------------------------------------------------------
// Every token group's counts and ranks are in global memory once all CTAs
// pass a grid-wide barrier (the launch is cooperative: all CTAs are
// resident).  Self-resetting: each CTA reads the generation word, then
// arrives; the last to arrive zeroes the count and bumps the generation,
// which the others wait for (bounded).  Then this CTA's share of the scatter
// reuses its shared memory (base: the CTA's dynamic shared memory, 1024-byte
// aligned).
__device__ __forceinline__ void fused_scatter_tail(const RouteArgs &a, unsigned char *base, int grp) {
  __syncthreads();
  // Grid-wide barrier (self-resetting, bounded): thread 0 arrives; the last
  // arrival resets the count and bumps the generation the others wait for.
  // Between its arrival and that wait, the CTA stages its token rows when
  // they are its own token group's (written by its cluster, visible since
  // the cluster barrier that ended the routing).
  __shared__ int passed, g0_s, last_s;
  if (threadIdx.x == 0) {
    int *gen = a.bar + 32;
    const int g0 = ld_acquire_s32(gen);
    g0_s = g0;
    passed = 1;
    last_s = atom_add_release_s32(a.bar, 1) == (int)gridDim.x - 1;  // releases this CTA's counts and ranks
    if (last_s) {
      // every CTA's writes are visible to the last arrival (the arrivals
      // released them); reset the count, then release the generation
      asm volatile("fence.acq_rel.gpu;\n" ::: "memory");
      *(volatile int *)a.bar = 0;
      st_release_s32(gen, g0 + 1);
    }
  }
  unsigned char *stage = a.sc.stage_bytes ? base + scatter_tab_bytes(a.sc.ng, a.sc.E, a.sc.per) : nullptr;
  int t_lo, n_tok;
  scatter_tokens(a.sc, blockIdx.x, &t_lo, &n_tok);
  const bool early = stage && n_tok > 0 && t_lo / kRouteTok == grp && (t_lo + n_tok - 1) / kRouteTok == grp &&
                     scatter_stage_bytes(n_tok, a.sc.d, a.sc.fp8) <= (size_t)a.sc.stage_bytes;
  if (early) scatter_stage_rows(a.sc, t_lo, n_tok, (uint4 *)stage);
  if (threadIdx.x == 0 && !last_s) {
    const int *gen = a.bar + 32;
    const long long c0 = clock64();
    while (ld_acquire_s32(gen) == g0_s) {
      if (clock64() - c0 > tc::kWaitCycles) {
        if (a.err) atomicExch(a.err, 55);
        passed = 0;  // counts may be incomplete: leave the scatter undone
        break;
      }
    }
    // acquired: the generation by ld.acquire, or (the last arrival) by the
    // fence after its count; the CTA barrier below passes it to the CTA
  }
  __syncthreads();
  pdl_trigger();
  if (!passed) return;
  __shared__ int warp_tot[kScatThreads / 32];
  scatter_block(a.sc, blockIdx.x, (int *)base, warp_tot, stage, (size_t)a.sc.stage_bytes, early);
}

template <bool NORM>
__global__ void __launch_bounds__(kRouteThreads, 1)
    route_kernel(const __grid_constant__ CUtensorMap tx, RouteArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const RouteSmem L = route_smem(a.S, a.nk_max, a.stages, a.m_tiles);
  uint64_t *full = (uint64_t *)(base + L.bars_off);
  uint64_t *empty = full + 8;
  uint64_t *xbar = empty + 8;  // B operand loaded by TMA (no norm)
  uint64_t *accb = xbar + 1;
  uint64_t *rbar = accb + 1;  // peers' partial logits received
  uint32_t *tmem_slot = (uint32_t *)(rbar + 1);
  volatile int *abort = (volatile int *)(tmem_slot + 1);
  int *flag = (int *)(tmem_slot + 2);  // [2] k-tiles loaded (the producer's own count)
  unsigned char *wring = base + L.w_off, *xs = base + L.x_off;
  float *part = (float *)(base + L.part_off), *logit = (float *)(base + L.logit_off);
  float *ss = (float *)(base + L.ss_off);
  int *cnt = (int *)(base + L.cnt_off);  // this CTA's pairs per expert
  int *pid = (int *)(base + L.pid_off);  // this CTA's pairs' experts

  // The S CTAs of a token group exchange through distributed shared memory:
  // a launch without S-CTA clusters returns at once (every CTA sees the same
  // size), leaving the scatter and the grid barrier untouched.
  if (cluster_ctas() != (uint32_t)a.S) {
    if (threadIdx.x == 0 && a.err) atomicExch(a.err, kShapeErrorBase + 3);
    return;
  }
  const int S = a.S, z = (int)(blockIdx.x % S), grp = (int)(blockIdx.x / S);
  const int t0 = grp * kRouteTok, ep = a.m_tiles * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = a.d / 64;
  const int kb = KT * z / S, ke = KT * (z + 1) / S, nk = ke - kb;
  const int stages = a.stages;
  const uint32_t stage_bytes = (uint32_t)a.m_tiles * kWBox;
  // Four accumulators per 128-expert tile (the K16 steps of a k-tile go
  // round-robin): dependent MMAs into one accumulator serialise, four short
  // chains overlap.  128 or 256 columns.
  constexpr int kAcc = 4;
  const uint32_t tcols = a.m_tiles * kAcc * kRouteTok;
  for (int e = threadIdx.x; e < ep; e += kRouteThreads) cnt[e] = 0;

  const int err_seen = threadIdx.x == 0 ? ld_err_word(a.err) : 0;
  if (threadIdx.x == 0) {
    *abort = 0;
    for (int s = 0; s < stages; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, kAcc);  // one commit per MMA issuer
    }
    tc::mbar_init(accb, kAcc);
    tc::mbar_init(xbar, 1);
    tc::mbar_init(rbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     tc::smem_u32(tmem_slot)),
                 "r"(tcols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  __syncwarp();  // lone-thread roles above: reconverge before the CTA-wide barrier
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  // Weights never change: the first ring fill starts before the wait on the
  // kernel that produced this layer's activations.
  // When the ring holds the whole K slice, all of it arrives on one barrier
  // phase: copies in flight together, one wait (a barrier phase per stage
  // paces the copies one after another).
  const int pre = min(stages, nk);
  const bool one_phase = nk <= stages;
  if (threadIdx.x == 0) {
    if (one_phase) tc::mbar_expect_tx(full, (uint32_t)nk * a.E * 128);
    for (int i = 0; i < pre; ++i)
      load_w_tile(a.wr, a.E, KT, a.m_tiles, kb + i, wring + (size_t)i * stage_bytes, one_phase ? full : full + i,
                  !one_phase);
  }
  // Norm: kTokThreads threads per token; thread `sub` owns the float4
  // columns c4b + kTokThreads u of the CTA's slice.  The gain is a weight:
  // its slice is loaded before the wait as well.
  const int tt = threadIdx.x / kTokThreads, sub = threadIdx.x % kTokThreads, tn = t0 + tt;
  const int c4b = kb * 16 + sub, c4e = ke * 16;
  float4 gv[kNormRegs], hv[kNormRegs];
  if (NORM) {
    const float4 *g4 = (const float4 *)a.gain;
#pragma unroll
    for (int u = 0; u < kNormRegs; ++u) {
      const int c = c4b + kTokThreads * u;
      gv[u] = c < c4e ? g4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  pdl_wait();
  if (!a.fuse) pdl_trigger();  // fused: the expert FFN may launch only once the scatter's barrier is passed
  if (threadIdx.x == 0 && err_seen) *abort = 1;  // an earlier timeout

  if (NORM) {
    const float4 *row = (const float4 *)(a.h + (size_t)(tn < a.T ? tn : 0) * a.d);
    const bool live = tn < a.T;
#pragma unroll
    for (int u = 0; u < kNormRegs; ++u) {
      const int c = c4b + kTokThreads * u;
      hv[u] = live && c < c4e ? row[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float acc = 0.0f;
#pragma unroll
    for (int u = 0; u < kNormRegs; ++u)
      acc += hv[u].x * hv[u].x + hv[u].y * hv[u].y + hv[u].z * hv[u].z + hv[u].w * hv[u].w;
    for (int c = c4b + kTokThreads * kNormRegs; live && c < c4e; c += kTokThreads) {  // wider slices
      const float4 v = row[c];
      acc += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
#pragma unroll
    for (int off = kTokThreads / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (sub == 0) ss[tt] = acc;
    tc::cluster_sync();
    float pv[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) pv[q] = q < S ? ld_cluster_f32(tc::cluster_addr(tc::smem_u32(ss + tt), q)) : 0.0f;
    float tot = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) tot += pv[q];  // rank order; every CTA of the cluster adds alike
    const float inv = rsqrtf(tot / a.d + a.eps);
    const float4 *g4 = (const float4 *)a.gain;
    for (int c = c4b, u = 0; c < c4e; c += kTokThreads, ++u) {
      float4 v, g;
      if (u < kNormRegs) {
#pragma unroll
        for (int q = 0; q < kNormRegs; ++q)
          if (q == u) {
            v = hv[q];
            g = gv[q];
          }
      } else {
        v = live ? row[c] : make_float4(0.f, 0.f, 0.f, 0.f);
        g = g4[c];
      }
      uint2 packed = make_uint2(0u, 0u);
      if (live) {
        __nv_bfloat162 p0 = __floats2bfloat162_rn(v.x * inv * g.x, v.y * inv * g.y);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(v.z * inv * g.z, v.w * inv * g.w);
        packed.x = *(uint32_t *)&p0;
        packed.y = *(uint32_t *)&p1;
        *(uint2 *)(a.xn + (size_t)tn * a.d + 4 * c) = packed;
      }
      // 128-byte swizzled K-major B tile: row tt, 16-byte chunk (col / 8) ^ (tt % 8)
      const int cl = 4 * c - kb * 64, kt = cl >> 6, col = cl & 63;
      const uint32_t off = (uint32_t)kt * kXBox + tt * 128 + ((((col >> 3) ^ (tt & 7)) << 4) | ((col & 7) * 2));
      *(uint2 *)(xs + off) = packed;
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  } else if (threadIdx.x == 0) {
    tc::mbar_expect_tx(xbar, (uint32_t)nk * kXBox);
    for (int i = 0; i < nk; ++i) tc::tma_load_2d(xs + (size_t)i * kXBox, &tx, (kb + i) * 64, t0, xbar);
  }
  __syncwarp();
  __syncthreads();

  if (threadIdx.x == 0) {  // producer: the rest of the K slice, if the ring is shorter
    int i = pre;
    for (; i < nk; ++i) {
      const int s = i % stages;
      if (!tc::mbar_wait(empty + s, ((i / stages) - 1) & 1, a.err, 51, abort)) break;
      load_w_tile(a.wr, a.E, KT, a.m_tiles, kb + i, wring + (size_t)s * stage_bytes, full + s);
    }
    flag[2] = i;
  } else if (lane == 0 && warp >= 1 && warp <= kAcc) {
    // MMA issuers: one thread per accumulator (K16 step k16 of every k-tile):
    // a single thread issuing N = 32 MMAs back to back waits on each issue.
    const int k16 = warp - 1;
    bool ok = NORM || tc::mbar_wait(xbar, 0, a.err, 52, abort);
    constexpr uint32_t idesc = tc::idesc_bf16(128, kRouteTok);
    for (int i = 0; i < nk && ok; ++i) {
      const int s = i % stages;
      if ((!one_phase || i == 0) && !tc::mbar_wait(one_phase ? full : full + s, one_phase ? 0 : (i / stages) & 1, a.err, 53, abort))
        break;
      tc::fence_after();
      const uint32_t xa = tc::smem_u32(xs + (size_t)i * kXBox);
      for (int mt = 0; mt < a.m_tiles; ++mt) {
        const uint32_t wa = tc::smem_u32(wring + (size_t)s * stage_bytes + mt * kWBox);
        tc::mma_bf16(tmem + (mt * kAcc + k16) * kRouteTok, tc::sw128_desc(wa) + 2 * k16, tc::sw128_desc(xa) + 2 * k16,
                     idesc, i != 0);
      }
      if (!one_phase) tc::mma_commit(empty + s);  // frees the stage for a refill
    }
    tc::mma_commit(accb);  // always: with no MMA issued (an abort) it arrives at once
  }
  __syncwarp();  // lone-thread roles above: reconverge before the CTA-wide barrier
  __syncthreads();

  // Partial logits: warp w drains TMEM lanes 32 (w % 4) .. of 128-expert tile w / 4.
  {
    const int mt = warp >> 2, q = warp & 3;
    const int e = mt * 128 + q * 32 + lane;
    uint32_t r[kRouteTok];
    bool have = false;
    if (mt < a.m_tiles) {
      // bounded, and waited for even after an abort: TMEM is freed only after the MMAs finished
      const long long c0 = clock64();
      while (!tc::mbar_try_wait(accb, 0) && clock64() - c0 < tc::kWaitCycles) {
      }
      tc::fence_after();
      const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + mt * kAcc * kRouteTok;
      tc::tmem_ld32(tl, r);
      tc::tmem_ld_wait(r);
#pragma unroll 1
      for (int acc = 1; acc < kAcc; ++acc) {  // fixed order: deterministic
        uint32_t r2[kRouteTok];
        tc::tmem_ld32(tl + acc * kRouteTok, r2);
        tc::tmem_ld_wait(r2);
#pragma unroll
        for (int t = 0; t < kRouteTok; ++t) r[t] = __float_as_uint(__uint_as_float(r[t]) + __uint_as_float(r2[t]));
      }
      have = !*abort;
    }
    if (mt < a.m_tiles) {
#pragma unroll
      for (int t = 0; t < kRouteTok; ++t) part[t * ep + e] = have ? __uint_as_float(r[t]) : 0.0f;
    }
  }
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // the bulk copies read part
  __syncwarp();
  tc::fence_before();
  __syncthreads();
  tc::cluster_sync();  // every CTA's partials are complete

  // CTA q reduces tokens [q tpr, (q + 1) tpr): every CTA sends those rows of
  // its partial to CTA q with one bulk shared-to-shared copy; the receiver
  // adds the S rows in rank order (deterministic).
  const int tpr = kRouteTok / S;  // tokens reduced by this CTA
  const uint32_t rows_bytes = (uint32_t)tpr * ep * 4;
  float *recv = (float *)(base + L.recv_off);
  if (threadIdx.x == 0) {
    if (S > 1) tc::mbar_expect_tx(rbar, (uint32_t)(S - 1) * rows_bytes);
    for (int q = 1; q < S; ++q) {
      const int j = (z + q) % S;
      tc::bulk_copy_to_peer(tc::cluster_addr(tc::smem_u32(recv) + (uint32_t)z * rows_bytes, (uint32_t)j),
                            tc::smem_u32(part + (size_t)j * tpr * ep), rows_bytes,
                            tc::cluster_addr(tc::smem_u32(rbar), (uint32_t)j));
    }
  }
  if (S > 1) {  // bounded, and waited for even after an abort: no copy may still target this CTA at exit
    const long long c0 = clock64();
    while (!tc::mbar_try_wait(rbar, 0)) {
      if (clock64() - c0 > tc::kWaitCycles) {
        if (threadIdx.x == 0 && a.err) atomicExch(a.err, 54);
        *abort = 1;
        break;
      }
    }
  }
  for (int idx = threadIdx.x; idx < tpr * ep; idx += kRouteThreads) {
    float sum = 0.0f;
    for (int q = 0; q < S; ++q)  // rank order
      sum += q == z ? part[(size_t)z * tpr * ep + idx] : recv[(size_t)q * tpr * ep + idx];
    logit[idx] = sum;
  }
  if (warp == 1) {
    tc::fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(tcols));
  }
  // Bounded drain of weight boxes still in flight after an abort.
  if (threadIdx.x == 0 && *abort) {
    for (int i = one_phase ? 0 : max(0, flag[2] - stages); i < (one_phase ? 1 : flag[2]); ++i) {
      const long long c0 = clock64();
      while (!tc::mbar_try_wait(full + i % stages, (i / stages) & 1) && clock64() - c0 < tc::kWaitCycles) {
      }
    }
    if (!NORM) {
      const long long c0 = clock64();
      while (!tc::mbar_try_wait(xbar, 0) && clock64() - c0 < tc::kWaitCycles) {
      }
    }
  }
  const int k = a.k, np = tpr * k;  // this CTA's pairs: tokens t0 + z tpr + j, slots s
  for (int j = warp; j < tpr; j += kRouteWarps) {
    const int t = t0 + z * tpr + j;
    if (t < a.T)
      topk_warp(logit + j * ep, a.E, k, lane, a.ids + (size_t)t * k, a.gates + (size_t)t * k, pid + j * k);
    else if (lane < k)
      pid[j * k + lane] = -1;
  }
  __syncwarp();
  __syncthreads();

  // Stable ranks: pair p of this CTA ranks after the earlier pairs of the CTA
  // with the same expert, then after those of the cluster's lower ranks.
  int my_e[kPairIters], my_rank[kPairIters];
#pragma unroll
  for (int u = 0; u < kPairIters; ++u) {
    const int p = threadIdx.x + u * kRouteThreads;
    my_e[u] = p < np ? pid[p] : -1;
    my_rank[u] = 0;
    if (my_e[u] >= 0) {
      for (int q = 0; q < p; ++q) my_rank[u] += pid[q] == my_e[u];
      atomicAdd(cnt + my_e[u], 1);
    }
  }
  __syncwarp();
  tc::cluster_sync();  // every CTA's expert counts are complete
#pragma unroll
  for (int u = 0; u < kPairIters; ++u) {
    if (my_e[u] < 0) continue;
    const uint32_t src = tc::smem_u32(cnt + my_e[u]);
    int pv[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) pv[q] = q < z ? ld_cluster_s32(tc::cluster_addr(src, q)) : 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) my_rank[u] += pv[q];
    a.rank[(size_t)(t0 + z * tpr) * k + threadIdx.x + u * kRouteThreads] = my_rank[u];
  }
  // The group's pairs per expert: CTA z writes experts z, z + S, ...
  for (int e = z + S * (int)threadIdx.x; e < a.E; e += S * kRouteThreads) {
    const uint32_t src = tc::smem_u32(cnt + e);
    int pv[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) pv[q] = q < S ? ld_cluster_s32(tc::cluster_addr(src, q)) : 0;
    int sum = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) sum += pv[q];
    a.gcount[(size_t)grp * a.E + e] = sum;
  }
  __syncwarp();
  tc::cluster_sync();  // peers' counts stay alive until every read is done
  if (a.fuse) fused_scatter_tail(a, base, grp);
}

template <bool NORM>
cudaError_t route_attributes() {
  static unsigned long long attr_set = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !((attr_set >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(route_kernel<NORM>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(route_kernel<NORM>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set |= 1ull << dev;
  }
  return cudaSuccess;
}

// Clusters of S CTAs (smem bytes of dynamic shared memory each) that can be
// resident at once: the cap on a cooperative launch, which must be decided
// before the launch (a refused launch would end a CUDA graph capture).
template <bool NORM>
int route_max_clusters(int S, uint32_t smem) {
  struct Entry {
    int dev, S;
    uint32_t smem;
    int n;
  };
  static Entry cache[16];
  static int n_cache = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  for (int i = 0; i < n_cache; ++i)
    if (cache[i].dev == dev && cache[i].S == S && cache[i].smem == smem) return cache[i].n;
  if (route_attributes<NORM>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, 1, 1);
  cfg.blockDim = dim3(kRouteThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, route_kernel<NORM>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (n_cache < 16) cache[n_cache++] = Entry{dev, S, smem, n};
  return n;
}

template <bool NORM>
cudaError_t launch_route(const CUtensorMap &tx, RouteArgs a, cudaStream_t st) {
  const RouteSmem L = route_smem(a.S, a.nk_max, a.stages, a.m_tiles);
  auto kern = route_kernel<NORM>;
  cudaError_t e = route_attributes<NORM>();
  if (e != cudaSuccess) return e;
  const int groups = ceil_div(a.T, kRouteTok);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.fuse ? a.grid : groups * a.S, 1, 1);
  cfg.blockDim = dim3(kRouteThreads, 1, 1);
  cfg.dynamicSmemBytes = L.bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[3];
  int na = 0;
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = a.S;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (a.fuse) {  // the CTAs wait on one another at the scatter's barrier: all must be resident
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, tx, a);
}

int num_sms_route();

cudaError_t route_common(bool norm, const float *h, const float *gain, float eps, bf16 *xn, const bf16 *wr,
                         int T, int d, int E, int k, int *ids, float *gates, int *rank, int *gcount, int *err,
                         cudaStream_t st, const ScatArgs *fused = nullptr, int *bar = nullptr) {
  if (T < 0 || d < 64 || d % 64 || E < 1 || E > 256 || k < 1 || k > 16 || k > E) return cudaErrorInvalidValue;
  if (T == 0) return cudaSuccess;
  RouteArgs a = {};
  a.h = h;
  a.gain = gain;
  a.eps = eps;
  a.xn = xn;
  a.T = T;
  a.d = d;
  a.E = E;
  a.k = k;
  const int KT = d / 64;
  a.S = KT >= 8 ? 8 : KT >= 4 ? 4 : KT >= 2 ? 2 : 1;
  a.nk_max = ceil_div(KT, a.S);
  a.m_tiles = E > 128 ? 2 : 1;
  const RouteSmem base = route_smem(a.S, a.nk_max, 0, a.m_tiles);
  const int fit = (int)((kSmemBudget - (int)base.bytes) / (a.m_tiles * (int)kWBox));
  a.stages = min(8, min(a.nk_max, fit));
  if (a.stages < 1) return cudaErrorInvalidValue;  // the K slice's B operand does not fit: d too large
  a.ids = ids;
  a.gates = gates;
  a.rank = rank;
  a.gcount = gcount;
  a.err = err;
  a.wr = wr;
  if (fused) {
    a.fuse = 1;
    a.bar = bar;
    a.sc = *fused;
    const RouteSmem full = route_smem(a.S, a.nk_max, a.stages, a.m_tiles);
    // The routing clusters must all be resident together; if they cannot
    // be, the launch is not fused (decided here: a refused launch would end
    // a CUDA graph capture).
    const int max_clusters = norm ? route_max_clusters<true>(a.S, full.bytes) : route_max_clusters<false>(a.S, full.bytes);
    const int groups = ceil_div(T, kRouteTok);
    if (groups > max_clusters) return cudaErrorCooperativeLaunchTooLarge;
    a.grid = a.S * groups;
    a.sc.per = ceil_div(T * k, a.grid);
    const size_t tab = scatter_tab_bytes(a.sc.ng, E, a.sc.per), usable = full.bytes - 1024;
    if (tab > usable) return cudaErrorInvalidValue;
    a.sc.stage_bytes = (int)(usable - tab);
    // e4m3 rows are written from the staged rows only: without room, two launches
    if (a.sc.fp8 && scatter_stage_bytes(a.sc.per / k + 2, d, 1) > (size_t)a.sc.stage_bytes)
      return cudaErrorCooperativeLaunchTooLarge;
  }
  CUtensorMap tx{};  // the norm path writes the B operand itself
  if (norm) return launch_route<true>(tx, a, st);
  cudaError_t e;
  e = tmap_bf16_cached(&tx, xn, (uint64_t)T, (uint64_t)d, kRouteTok);
  if (e != cudaSuccess) return e;
  return launch_route<false>(tx, a, st);
}

int num_sms_route() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace

size_t moe_group_count_ints(int T, int E) { return (size_t)ceil_div(T, kRouteTok) * E; }

cudaError_t moe_norm_route(const float *h, const float *gain, float eps, bf16 *xn, const bf16 *wr, int T, int d,
                           int E, int k, int *ids, float *gates, int *rank, int *gcount, int *err,
                           cudaStream_t st) {
  return route_common(true, h, gain, eps, xn, wr, T, d, E, k, ids, gates, rank, gcount, err, st);
}

cudaError_t moe_route(const bf16 *xn, const bf16 *wr, int T, int d, int E, int k, int *ids, float *gates,
                      int *rank, int *gcount, int *err, cudaStream_t st) {
  return route_common(false, nullptr, nullptr, 0.0f, const_cast<bf16 *>(xn), wr, T, d, E, k, ids, gates, rank,
                      gcount, err, st);
}

namespace {

cudaError_t scatter_args(ScatArgs &a, const bf16 *xn, const int *ids, const int *gcount, int *slot_row, int T,
                         int d, int E, int k, int tile_rows, bf16 *x_tiles, int *offs, int *work, int *n_work,
                         int max_work, unsigned long long *stats, const Fp8Experts *fp8) {
  if (fp8 && (d % 128 || !fp8->kx)) return cudaErrorInvalidValue;
  if (T < 0 || d % 64 || E < 1 || E > kScatThreads || k < 1 || tile_rows != 128) return cudaErrorInvalidValue;
  if ((size_t)max_work < moe_max_work(T, k, E, tile_rows)) return cudaErrorInvalidValue;
  a.xn = xn;
  a.ids = ids;
  a.gcount = gcount;
  a.slot_row = slot_row;
  a.x_tiles = x_tiles;
  a.T = T;
  a.d = d;
  a.E = E;
  a.k = k;
  a.tile_rows = tile_rows;
  a.ng = ceil_div(T, kRouteTok);
  a.offs = offs;
  a.work = work;
  a.n_work = n_work;
  a.sync = work + 2 * max_work;
  a.max_work = max_work;
  a.stats = stats;
  a.stage_bytes = 0;
  a.fp8 = fp8 ? 1 : 0;
  a.kx = fp8 ? fp8->kx : nullptr;
  return cudaSuccess;
}

}  // namespace

cudaError_t moe_scatter(const bf16 *xn, const int *ids, const int *gcount, int *slot_row, int T, int d, int E,
                        int k, int tile_rows, bf16 *x_tiles, int *offs, int *work, int *n_work, int max_work,
                        cudaStream_t st, unsigned long long *stats, const Fp8Experts *fp8) {
  ScatArgs a;
  cudaError_t e = scatter_args(a, xn, ids, gcount, slot_row, T, d, E, k, tile_rows, x_tiles, offs, work, n_work,
                               max_work, stats, fp8);
  if (e != cudaSuccess) return e;
  const int TK = T * k;
  const int grid = max(1, min(ceil_div(TK, 2 * (kScatThreads / 32)), 2 * num_sms_route()));
  a.per = ceil_div(TK, grid);
  const size_t tab = scatter_tab_bytes(a.ng, E, a.per);
  if (tab > 200 * 1024) return cudaErrorInvalidValue;
  // room for the block's token rows (at most per / k + 2 of them), if it fits
  const size_t stage = scatter_stage_bytes(a.per / k + 2, d, a.fp8);
  a.stage_bytes = tab + stage <= 200 * 1024 ? (int)stage : 0;
  if (a.fp8 && !a.stage_bytes) return cudaErrorInvalidValue;  // e4m3 rows are written from the staged rows
  const size_t smem = tab + a.stage_bytes;
  static unsigned long long attr_set = 0;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !((attr_set >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set |= 1ull << dev;
  }
  return launch_pdl(scatter_kernel, dim3(grid), dim3(kScatThreads), smem, st, a);
}

cudaError_t moe_route_scatter(const float *h, const float *gain, float eps, bf16 *xn, const bf16 *wr, int T, int d,
                              int E, int k, int *ids, float *gates, int *slot_row, int *gcount, bf16 *x_tiles,
                              int *offs, int *work, int *n_work, int max_work, int *bar, int *err, cudaStream_t st,
                              unsigned long long *stats, int *launches, const Fp8Experts *fp8) {
  const bool norm = h != nullptr;
  const int S = (d / 64) >= 8 ? 8 : (d / 64) >= 4 ? 4 : (d / 64) >= 2 ? 2 : 1;
  const int grid = ceil_div(T, kRouteTok) * S;
  // DG_FUSE_ROUTE=0 keeps the two launches (for profilers that replay one
  // kernel at a time: an Nsight Compute capture of the cooperative fused
  // launch faulted on the GB300).
  static const bool fuse_allowed = [] {
    const char *v = getenv("DG_FUSE_ROUTE");
    return !(v && v[0] == '0');
  }();
  if (fuse_allowed && bar && grid <= num_sms_route()) {  // one CTA per SM: every routing CTA can be resident
    ScatArgs a;
    cudaError_t e = scatter_args(a, xn, ids, gcount, slot_row, T, d, E, k, kExpertTileRows, x_tiles, offs, work,
                                 n_work, max_work, stats, fp8);
    if (e != cudaSuccess) return e;
    e = route_common(norm, h, gain, eps, xn, wr, T, d, E, k, ids, gates, slot_row, gcount, err, st, &a, bar);
    if (e != cudaErrorCooperativeLaunchTooLarge) {
      if (launches) *launches = 1;
      return e;
    }
    cudaGetLastError();  // too few clusters resident together for the routing: two launches
  }
  cudaError_t e = route_common(norm, h, gain, eps, xn, wr, T, d, E, k, ids, gates, slot_row, gcount, err, st);
  if (e != cudaSuccess) return e;
  if (launches) *launches = 2;
  return moe_scatter(xn, ids, gcount, slot_row, T, d, E, k, kExpertTileRows, x_tiles, offs, work, n_work, max_work,
                     st, stats, fp8);
}

}  // namespace dg
