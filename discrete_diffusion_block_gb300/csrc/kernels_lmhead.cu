// LM head fused with the vocabulary reduction of the sampler, as one
// persistent warp-specialised tcgen05 kernel.
//
// Work unit = (vocab tile of 256, block of 128 token rows).  One CTA per SM
// walks the units u = blockIdx.x, blockIdx.x + gridDim.x, ...; unit u covers
// vocab tile u / m_tiles and row block u % m_tiles, so the CTAs that share a
// vocab tile run it at the same time and its weights are read from HBM once.
//
//   warp 0 (one thread)  producer: per 64-wide K step the 128-row A tile
//                        (normalised rows, and the low half of their hi/lo
//                        split) and the two 128-row tiles of 256 W_out rows
//                        into a 3-stage ring; all operands are stored as
//                        operand tiles (tiled_index), so each is one
//                        contiguous bulk copy;
//   warp 1 (one thread)  allocates all 512 TMEM columns (two 128 x 256 fp32
//                        accumulators) and issues tcgen05.mma, unit n into
//                        accumulator n & 1;
//   warps 2-5, 6-9       two epilogue groups; group e drains accumulator e
//                        (units n = e, e + 2, ...) while the tensor core
//                        fills the other.  Thread = one token row, read
//                        straight from TMEM 32 columns at a time:
//                        row_tile_partial (sampler.cuh), the same code the
//                        standalone reduction of given logits runs: the
//                        canonical tile partials of the sampler; the logits
//                        never reach HBM (MODE 0).  MODE 1 writes the fp32
//                        logits instead, MODE 2 both, from one accumulator.
//
// Every wait is bounded (about a second); a wait that gives up records an
// error word and makes the CTA's later waits return at once.
#include <cuda.h>

#include "gemm_tc.cuh"
#include "internal.h"
#include "sampler.cuh"

namespace dg {

namespace {

constexpr int kLmStages = 3;
constexpr int kLmThreads = 320;
constexpr uint32_t kLmABytes = 128 * 128;  // 128 rows x 64 bf16
constexpr uint32_t kLmBBytes = 256 * 128;  // 256 rows x 64 bf16
constexpr int kLmAccCols = 256;

template <int NA>
struct LmSmem {
  static constexpr uint32_t stage_bytes = NA * kLmABytes + kLmBBytes;
  static constexpr size_t ring = (size_t)kLmStages * stage_bytes;
  // then: Gumbel bound table [256] floats; full[S], empty[S], acc_full[2],
  // acc_empty[2]; TMEM address and abort flag
  static constexpr size_t gtab = ring;
  static constexpr size_t bars = gtab + 256 * 4;
  static constexpr size_t bytes = bars + (2 * kLmStages + 4) * 8 + 16 + 1024;
};

// One token row of an accumulator in tensor memory, 32 columns per load.
struct TmemRowSrc {
  uint32_t taddr;  // lane (row) and first column of the row's 256 logits
  __device__ __forceinline__ void issue(int c, uint32_t *x) { tc::tmem_ld32(taddr + 32 * c, x); }
  __device__ __forceinline__ void wait(uint32_t *x) { tc::tmem_ld_wait(x); }
};

struct LmArgs {
  const bf16 *xn, *xn_lo;   // normalised rows (hi, lo) as operand tiles of [T][K]
  const bf16 *w;            // W_out as operand tiles of [V][K]
  int T, V, K;              // token rows, vocabulary, model width
  PartialPlanes P;          // partials planes [T][V/256] (modes 0, 2)
  float *logits;            // [T][V] fp32 (modes 1, 2)
  uint32_t ctr2, key0, key1;
  float inv_tau;            // 1 / temperature of the re-noise keys
  int rows_per_req;         // > 0: row r is position r % rows_per_req of request r / rows_per_req,
                            // whose Gumbel stream is keyed by the sample seed + request
  const StepParams *dyn;    // when set, the stream words and inv_tau come from device memory
  int *err;
};

// MODE 0: sampler partials; MODE 1: fp32 logits; MODE 2: both, from the same
// accumulator (so that the partials can be checked on the logits they came from).
template <int NA, int MODE>
__global__ void __launch_bounds__(kLmThreads, 1) lm_head_kernel(LmArgs g) {
  using S = LmSmem<NA>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  float *gbound = (float *)(base + S::gtab);
  uint64_t *full = (uint64_t *)(base + S::bars);
  uint64_t *empty = full + kLmStages;
  uint64_t *acc_full = empty + kLmStages;
  uint64_t *acc_empty = acc_full + 2;
  uint32_t *tmem_slot = (uint32_t *)(acc_empty + 2);
  volatile int *abort = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = ceil_div(g.T, 128), tiles = g.V / kVocabTile;
  const int n_units = m_tiles * tiles, KT = g.K / tc::kBK;
  if ((int)blockIdx.x >= n_units) return;

  const int err_seen = threadIdx.x == 0 ? ld_err_word(g.err) : 0;
  if (threadIdx.x == 0) {
    *abort = 0;
    for (int s = 0; s < kLmStages; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(acc_full + b, 1);
      tc::mbar_init(acc_empty + b, 4);  // one arrival per epilogue warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  if (MODE != 1 && threadIdx.x >= 64)
    for (int b = threadIdx.x - 64; b < 256; b += kLmThreads - 64) gbound[b] = gumbel_bucket_bound(b);
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     tc::smem_u32(tmem_slot)),
                 "r"((uint32_t)(2 * kLmAccCols)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  __syncwarp();  // lone-thread roles above: reconverge before the CTA-wide barrier
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  auto a_tile = [&](int s, int h) { return base + (size_t)s * S::stage_bytes + h * kLmABytes; };
  auto b_tile = [&](int s) { return base + (size_t)s * S::stage_bytes + NA * kLmABytes; };
  // A tile of row block mt (the last block may be partial: its rows past T
  // stay stale in shared memory, and their accumulator rows are never
  // stored); the 256 W_out rows of vocab tile v as two full 128-row tiles.
  auto a_bytes = [&](int mt) { return (uint32_t)min(128, g.T - 128 * mt) * 128; };
  auto load_a = [&](int s, int mt, int kt) {
    tc::bulk_load(a_tile(s, 0), g.xn + tiled_index(g.T, g.K, 128 * mt, 64 * kt), a_bytes(mt), full + s);
    if (NA == 2)
      tc::bulk_load(a_tile(s, 1), g.xn_lo + tiled_index(g.T, g.K, 128 * mt, 64 * kt), a_bytes(mt), full + s);
  };
  auto load_b = [&](int s, int v, int kt) {
    for (int h = 0; h < 2; ++h)
      tc::bulk_load(b_tile(s) + h * 16384, g.w + tiled_index(g.V, g.K, kVocabTile * v + 128 * h, 64 * kt), 16384u,
                    full + s);
  };

  // The weights never change: the first unit's W_out tiles are requested
  // before waiting for the kernel that produced the normalised rows.
  const int pre = min(kLmStages, KT);
  if (warp == 0 && lane == 0) {
    const int v = blockIdx.x / m_tiles, mt = blockIdx.x - v * m_tiles;
    for (int i = 0; i < pre; ++i) {
      tc::mbar_expect_tx(full + i, NA * a_bytes(mt) + kLmBBytes);
      load_b(i, v, i);
    }
  }
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0 && err_seen) *abort = 1;

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int v = u / m_tiles, mt = u - v * m_tiles;
        for (int kt = 0; kt < KT; ++kt, ++it) {
          const int s = it % kLmStages, r = it / kLmStages;
          if (r > 0) tc::mbar_wait(empty + s, (r - 1) & 1, g.err, 11, abort);
          if (*abort) break;
          if (it >= pre) {
            tc::mbar_expect_tx(full + s, NA * a_bytes(mt) + kLmBBytes);
            load_b(s, v, kt);
          }
          load_a(s, mt, kt);
        }
        if (*abort) break;
      }
      if (*abort) {  // drain the copies still in flight (bounded)
        for (int i = it - 1; i >= 0 && i >= it - kLmStages; --i) {
          const long long t0 = clock64();
          while (!tc::mbar_try_wait(full + i % kLmStages, (i / kLmStages) & 1) &&
                 clock64() - t0 < tc::kWaitCycles) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16(128, kLmAccCols);
      int it = 0, n = 0;
      for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++n) {
        const int buf = n & 1;
        if (n >= 2) tc::mbar_wait(acc_empty + buf, ((n >> 1) - 1) & 1, g.err, 12, abort);
        tc::fence_after();
        const uint32_t d_tmem = tmem + buf * kLmAccCols;
        for (int kt = 0; kt < KT; ++kt, ++it) {
          const int s = it % kLmStages, r = it / kLmStages;
          tc::mbar_wait(full + s, r & 1, g.err, 13, abort);
          tc::fence_after();
          const uint64_t bdesc = tc::sw128_desc(tc::smem_u32(b_tile(s)));
#pragma unroll
          for (int h = 0; h < NA; ++h) {
            const uint64_t adesc = tc::sw128_desc(tc::smem_u32(a_tile(s, h)));
#pragma unroll
            for (int kk = 0; kk < tc::kBK / 16; ++kk)
              tc::mma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kt | kk | h) ? 1u : 0u);
          }
          tc::mma_commit(empty + s);
        }
        tc::mma_commit(acc_full + buf);
      }
    }
  } else {
    // ---- epilogue groups ---------------------------------------------------
    const int e = (warp - 2) >> 2;   // group: accumulator e
    const int q = warp & 3;          // TMEM lane quarter this warp may read
    const int row = 32 * q + lane;   // token row inside the unit
    uint32_t c2 = g.ctr2, k0 = g.key0, k1 = g.key1;
    float inv_tau = g.inv_tau;
    if (g.dyn) {
      c2 = g.dyn->ctr2;
      k0 = g.dyn->key0;
      k1 = g.dyn->key1;
      inv_tau = g.dyn->inv_tau;
    }
    int n = e;
    for (int u = blockIdx.x + e * gridDim.x; u < n_units; u += 2 * gridDim.x, n += 2) {
      const int v = u / m_tiles, mt = u - v * m_tiles;
      const int pos = mt * 128 + row;
      tc::mbar_wait(acc_full + e, (n >> 1) & 1, g.err, 14, abort);
      tc::fence_after();
      const uint32_t taddr = tmem + e * kLmAccCols + ((uint32_t)(32 * q) << 16);
      if (MODE != 0) {
        float *dst = g.logits + (size_t)pos * g.V + (size_t)v * kVocabTile;
#pragma unroll 1
        for (int c = 0; c < kLmAccCols / 32; ++c) {
          uint32_t x[32];
          tc::tmem_ld32(taddr + 32 * c, x);
          tc::tmem_ld_wait(x);
          if (pos < g.T) {
            float4 *d4 = (float4 *)(dst + 32 * c);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              d4[j] = make_float4(__uint_as_float(x[4 * j]), __uint_as_float(x[4 * j + 1]),
                                  __uint_as_float(x[4 * j + 2]), __uint_as_float(x[4 * j + 3]));
          }
        }
      }
      Partial p{};
      if (MODE != 1) {
        TmemRowSrc src{taddr};
        const int b = g.rows_per_req > 0 ? pos / g.rows_per_req : 0;
        const uint64_t seed = (((uint64_t)k1 << 32) | k0) + (uint64_t)b;
        p = row_tile_partial(src, v, (uint32_t)(pos - b * g.rows_per_req), c2, (uint32_t)seed,
                             (uint32_t)(seed >> 32), gbound, inv_tau);
      }
      // the accumulator is free for unit n + 2
      tc::fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(acc_empty + e)) : "memory");
      if (MODE != 1 && pos < g.T) {
        const size_t o = (size_t)pos * tiles + v;
        g.P.m[o] = p.m;
        g.P.a[o] = p.a;
        g.P.s[o] = p.s;
        g.P.gk[o] = p.gk;
        g.P.gi[o] = p.gi;
      }
    }
  }
  __syncwarp();  // lone-thread roles above: reconverge before the CTA-wide barrier
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                 "r"((uint32_t)(2 * kLmAccCols)));
  }
}

int lm_num_sms() {
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

template <int NA, int MODE>
cudaError_t launch_lm_head(const LmArgs &g, cudaStream_t st) {
  using S = LmSmem<NA>;
  static_assert(S::bytes <= 232448, "shared memory of the LM head");
  auto kern = lm_head_kernel<NA, MODE>;
  static unsigned long long attr_set = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !((attr_set >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::bytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set |= 1ull << dev;
  }
  const int m_tiles = ceil_div(g.T, 128), units = m_tiles * (g.V / kVocabTile);
  // a multiple of m_tiles, so that each CTA keeps one row block and the CTAs
  // sharing a vocab tile run together
  int grid = lm_num_sms() / m_tiles * m_tiles;
  if (grid < m_tiles) grid = m_tiles;
  if (grid > units) grid = units;
  return launch_pdl(kern, dim3(grid), dim3(kLmThreads), S::bytes, st, g);
}

}  // namespace

static cudaError_t lm_head_launch(const bf16 *xn, const bf16 *xn_lo, const bf16 *w_out, int T, int d,
                                  int V, LmArgs &g, int mode, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (d % tc::kBK || V % kVocabTile) return cudaErrorInvalidValue;
  g.xn = xn;
  g.xn_lo = xn_lo;
  g.w = w_out;
  g.T = T;
  g.V = V;
  g.K = d;
  if (mode == 0) return xn_lo ? launch_lm_head<2, 0>(g, st) : launch_lm_head<1, 0>(g, st);
  if (mode == 2) return xn_lo ? launch_lm_head<2, 2>(g, st) : launch_lm_head<1, 2>(g, st);
  return xn_lo ? launch_lm_head<2, 1>(g, st) : launch_lm_head<1, 1>(g, st);
}

cudaError_t gemm_lm_head_partials(const bf16 *xn, const bf16 *xn_lo, const bf16 *w_out, int T, int d,
                                  int V, uint64_t seed, int canvas, int step, float inv_tau,
                                  void *partials, int *err, cudaStream_t st, const StepParams *dyn,
                                  float *logits, int rows_per_req) {
  LmArgs g{};
  g.inv_tau = inv_tau;
  g.rows_per_req = rows_per_req;
  g.P = PartialPlanes::at(partials, T, V / kVocabTile);
  g.logits = logits;
  g.ctr2 = gumbel_ctr2(canvas, step);
  g.key0 = (uint32_t)seed;
  g.key1 = (uint32_t)(seed >> 32);
  g.dyn = dyn;
  g.err = err;
  return lm_head_launch(xn, xn_lo, w_out, T, d, V, g, logits ? 2 : 0, st);
}

cudaError_t gemm_lm_head_logits(const bf16 *xn, const bf16 *xn_lo, const bf16 *w_out, int T, int d,
                                int V, float *logits, int *err, cudaStream_t st) {
  LmArgs g{};
  g.logits = logits;
  g.err = err;
  return lm_head_launch(xn, xn_lo, w_out, T, d, V, g, 1, st);
}

}  // namespace dg
