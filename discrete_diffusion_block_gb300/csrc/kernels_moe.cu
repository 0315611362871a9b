// Routed-expert feed-forward of one MoE layer as a single persistent
// warp-specialised tcgen05 kernel: for every routed expert e with token rows
// X_e (gathered in expert order),
//   act_e = SiLU(X_e Wg_e^T) * (X_e Wu_e^T)        (phase A, "gate/up")
//   y_e   = act_e Wd_e^T                           (phase B, "down")
//
// Units.  A work item is (expert, up to 128 of its rows).  Phase A units are
// (item, 128-row block of the interleaved gate/up weights) -- 64 gate rows
// and the matching 64 up rows, so SwiGLU is local to the tile; phase B units
// are (item, 128-row block of W_down).  All units sit in one list, phase A
// first; CTAs (one per SM) take the next unit from a global counter, so the
// small phase B units fill the tail of phase A and no SM idles while another
// still has a long queue.  A phase B unit needs the whole act row block of its
// item: its producer waits (bounded) until the item's phase A units have all
// published their outputs (per-item counter, release/acquire, then a proxy
// fence before the TMA reads them).
//
// Operands.  Expert weights and the item rows (gathered by moe_scatter, and
// the SwiGLU output written here by phase A) are stored as 16 KB tiles of 128
// rows x 64 columns already in the tensor core's swizzled shared-memory order,
// so each k-step of a unit stages its operands with two contiguous bulk
// copies (the weight tile, the item's valid rows) instead of row-by-row
// tensor copies.
//
// Roles (192 threads):
//   warp 4, one thread  -- takes units, hands them to the other roles through
//                          a 4-deep shared-memory queue, and streams A (one
//                          weight tile) and B (the item's rows) per k-step
//                          into a 6-stage ring;
//   warp 5, one thread  -- owns 2 x 128 TMEM columns and issues tcgen05.mma
//                          (M = 128, N = rows rounded up to 16), unit n into
//                          accumulator n & 1;
//   warps 0-3           -- drain accumulator n & 1 into an fp32 tile and run
//                          the SwiGLU (A) or store (B) epilogue while the
//                          tensor core already works on the next unit.
// Every wait is bounded; a wait that gives up records an error word and makes
// the CTA's later waits return at once.
#include <cuda.h>

#include "gemm_tc.cuh"
#include "internal.h"

namespace dg {

namespace {

constexpr int kFfnStages = 6;
constexpr int kFfnThreads = 192;
constexpr int kFfnBN = kExpertTileRows;  // rows per item = MMA N upper bound
constexpr int kFfnQueue = 4;
constexpr uint32_t kFfnABytes = 128 * 128;
constexpr uint32_t kFfnBBytes = kFfnBN * 128;
constexpr uint32_t kFfnStageBytes = kFfnABytes + kFfnBBytes;
constexpr int kFfnEpiCols = 64;            // accumulator columns (rows of the item) per epilogue pass
constexpr int kFfnLdc = kFfnEpiCols + 1;

struct FfnSmem {
  static constexpr size_t ring = (size_t)kFfnStages * kFfnStageBytes;
  static constexpr size_t tile = ring;                                   // fp32 [128][kFfnLdc]: 64 columns at a time
  static constexpr size_t queue = tile + (size_t)128 * kFfnLdc * 4;      // UnitInfo [kFfnQueue]
  static constexpr size_t bars = (queue + kFfnQueue * 32 + 15) & ~(size_t)15;
  // full[S], empty[S], acc_full[2], acc_empty[2], q_full[Q], q_empty[Q]; TMEM address; abort flag
  static constexpr size_t bytes = bars + (2 * kFfnStages + 4 + 2 * kFfnQueue) * 8 + 16 + 1024;
};

struct UnitInfo {
  int u;        // unit index, -1 = no more units
  int phase;    // 0: gate/up, 1: down
  int item, mt, b_row, n_valid, e, pad;
};

// Operands are stored as 16 KB tiles (128 rows x 64 columns, in the
// tensor core's 128-byte swizzled shared-memory order), [row block][k-tile];
// one contiguous bulk copy moves a weight tile, one moves the valid rows of
// an item's tile.
struct FfnArgs {
  const int *work, *n_work, *offs;
  const bf16 *wgu, *wd;  // [E][2F/128][d/64] and [E][d/128][F/64] tiles
  const bf16 *x;         // [item][d/64] tiles: the item's token rows
  int *done;   // [max_work] phase A units finished per item
  int *next;   // unit counter
  int E, d, F;
  bf16 *act;   // [item][F/64] tiles: SwiGLU output rows
  float *y;    // [rows][d]
  int *err;
};

constexpr int kTileElems = 128 * 64;

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   tc::smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;\n" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(b)) : "memory");
}

__device__ __forceinline__ float swiglu_f(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

__global__ void __launch_bounds__(kFfnThreads, 1) moe_ffn_kernel(FfnArgs g) {
  using S = FfnSmem;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  float *tile = (float *)(base + S::tile);
  UnitInfo *queue = (UnitInfo *)(base + S::queue);
  uint64_t *full = (uint64_t *)(base + S::bars);
  uint64_t *empty = full + kFfnStages;
  uint64_t *acc_full = empty + kFfnStages;
  uint64_t *acc_empty = acc_full + 2;
  uint64_t *q_full = acc_empty + 2;
  uint64_t *q_empty = q_full + kFfnQueue;
  uint32_t *tmem_slot = (uint32_t *)(q_empty + kFfnQueue);
  volatile int *abort = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    *abort = 0;
    for (int s = 0; s < kFfnStages; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(acc_full + b, 1);
      tc::mbar_init(acc_empty + b, 4);  // one arrival per epilogue warp
    }
    for (int q = 0; q < kFfnQueue; ++q) {
      tc::mbar_init(q_full + q, 1);
      tc::mbar_init(q_empty + q, 2);  // the MMA thread and the epilogue
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     tc::smem_u32(tmem_slot)),
                 "r"((uint32_t)(2 * kFfnBN)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  __syncwarp();  // lone-thread roles above: reconverge before the CTA-wide barrier
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the work list and the gathered rows come from earlier kernels
  pdl_trigger();
  if (threadIdx.x == 0 && g.err && *(volatile int *)g.err) *abort = 1;

  const int n_items = *g.n_work;
  const int mA = (2 * g.F) / 128, mB = g.d / 128;
  const int nA = n_items * mA, n_units = nA + n_items * mB;
  const int KTA = g.d / tc::kBK, KTB = g.F / tc::kBK;
  auto a_tile = [&](int s) { return base + (size_t)s * kFfnStageBytes; };
  auto b_tile = [&](int s) { return base + (size_t)s * kFfnStageBytes + kFfnABytes; };

  if (warp == 4) {
    if (lane == 0) {
      int it = 0;
      for (int n = 0;; ++n) {
        const int q = n % kFfnQueue;
        if (n >= kFfnQueue) tc::mbar_wait(q_empty + q, ((n / kFfnQueue) - 1) & 1, g.err, 21, abort);
        const int u = *abort ? n_units : atomicAdd(g.next, 1);
        UnitInfo inf;
        inf.u = u < n_units ? u : -1;
        if (inf.u >= 0) {
          inf.phase = u >= nA;
          const int v = inf.phase ? u - nA : u, per = inf.phase ? mB : mA;
          inf.item = v / per;
          inf.mt = v - inf.item * per;
          const int e = g.work[2 * inf.item], n0 = g.work[2 * inf.item + 1];
          const int e0 = g.offs[e];
          inf.b_row = e0 + n0;
          inf.n_valid = min(kFfnBN, g.offs[e + 1] - e0 - n0);
          inf.e = e;
        }
        queue[q] = inf;
        mbar_arrive(q_full + q);  // release: the entry is visible to the waiting roles
        if (inf.u < 0) break;
        const int KT = inf.phase ? KTB : KTA;
        const bf16 *asrc = inf.phase ? g.wd + (size_t)(inf.e * mB + inf.mt) * KTB * kTileElems
                                     : g.wgu + (size_t)(inf.e * mA + inf.mt) * KTA * kTileElems;
        const bf16 *bsrc = (inf.phase ? g.act : g.x) + (size_t)inf.item * KT * kTileElems;
        const uint32_t b_bytes = (uint32_t)((inf.n_valid + 7) & ~7) * 128;  // the item's valid rows
        const uint32_t tx = kFfnABytes + b_bytes;
        if (inf.phase) {
          // the item's act rows: every phase A unit of it must have published
          const long long t0 = clock64();
          while (ld_acquire(g.done + inf.item) < mA) {
            if (*abort) break;
            if (clock64() - t0 > tc::kWaitCycles) {
              if (g.err) atomicExch(g.err, 22);
              *abort = 1;
              break;
            }
          }
          asm volatile("fence.proxy.async.global;\n" ::: "memory");
        }
        for (int kt = 0; kt < KT; ++kt, ++it) {
          const int s = it % kFfnStages, r = it / kFfnStages;
          if (r > 0) tc::mbar_wait(empty + s, (r - 1) & 1, g.err, 23, abort);
          if (*abort) break;
          tc::mbar_expect_tx(full + s, tx);
          bulk_load(a_tile(s), asrc + (size_t)kt * kTileElems, kFfnABytes, full + s);
          bulk_load(b_tile(s), bsrc + (size_t)kt * kTileElems, b_bytes, full + s);
        }
        if (*abort) {  // drain the copies in flight (bounded), then hand over the end marker
          for (int i = it - 1; i >= 0 && i >= it - kFfnStages; --i) {
            const long long t0 = clock64();
            while (!tc::mbar_try_wait(full + i % kFfnStages, (i / kFfnStages) & 1) &&
                   clock64() - t0 < tc::kWaitCycles) {
            }
          }
        }
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      int it = 0;
      for (int n = 0;; ++n) {
        const int q = n % kFfnQueue;
        tc::mbar_wait(q_full + q, (n / kFfnQueue) & 1, g.err, 24, abort);
        const UnitInfo inf = queue[q];
        if (inf.u < 0 || *abort) break;
        const int buf = n & 1;
        if (n >= 2) tc::mbar_wait(acc_empty + buf, ((n >> 1) - 1) & 1, g.err, 25, abort);
        tc::fence_after();
        const uint32_t d_tmem = tmem + buf * kFfnBN;
        const uint32_t idesc = tc::idesc_bf16(128, max(16, (inf.n_valid + 15) & ~15));
        const int KT = inf.phase ? KTB : KTA;
        for (int kt = 0; kt < KT; ++kt, ++it) {
          const int s = it % kFfnStages, r = it / kFfnStages;
          tc::mbar_wait(full + s, r & 1, g.err, 26, abort);
          tc::fence_after();
          const uint64_t adesc = tc::sw128_desc(tc::smem_u32(a_tile(s)));
          const uint64_t bdesc = tc::sw128_desc(tc::smem_u32(b_tile(s)));
#pragma unroll
          for (int kk = 0; kk < tc::kBK / 16; ++kk)
            tc::mma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kt | kk) ? 1u : 0u);
          tc::mma_commit(empty + s);
        }
        tc::mma_commit(acc_full + buf);
        mbar_arrive(q_empty + q);
      }
    }
  } else {
    // ---- epilogue: warps 0-3, thread = accumulator row ------------------------
    const int row = threadIdx.x;
    for (int n = 0;; ++n) {
      const int q = n % kFfnQueue;
      tc::mbar_wait(q_full + q, (n / kFfnQueue) & 1, g.err, 27, abort);
      const UnitInfo inf = queue[q];
      if (inf.u < 0 || *abort) break;
      const int buf = n & 1;
      tc::mbar_wait(acc_full + buf, (n >> 1) & 1, g.err, 28, abort);
      tc::fence_after();
      const uint32_t trow = tmem + buf * kFfnBN + ((uint32_t)(warp * 32) << 16);
      // 64 accumulator columns (item rows) per pass through the fp32 tile
      for (int h0 = 0; h0 < inf.n_valid; h0 += kFfnEpiCols) {
        const int nh = min(kFfnEpiCols, inf.n_valid - h0);
        const int nchunks = (nh + 31) >> 5;
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
          uint32_t v[32];
          tc::tmem_ld32(trow + h0 + 32 * c, v);
          tc::tmem_ld_wait(v);
#pragma unroll
          for (int j = 0; j < 32; ++j) tile[row * kFfnLdc + 32 * c + j] = __uint_as_float(v[j]);
        }
        if (h0 + kFfnEpiCols >= inf.n_valid) {  // last pass: the accumulator is free for unit n + 2
          tc::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty + buf);
        }
        epi_sync();
        if (inf.phase == 0) {
          // SwiGLU: rows j and 64 + j hold the gate and up projections of
          // feature 64 * mt + j; each lane writes two adjacent features of an
          // item row into the act tile (item, k-tile mt) of the down GEMM.
          const int j = 2 * lane;
          unsigned char *blk = (unsigned char *)(g.act + ((size_t)inf.item * (g.F / 64) + inf.mt) * kTileElems);
          for (int tb = warp; tb < nh; tb += 16) {
            float g0[4], g1[4], u0[4], u1[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int t = min(tb + 4 * k, nh - 1);
              g0[k] = tile[j * kFfnLdc + t];
              g1[k] = tile[(j + 1) * kFfnLdc + t];
              u0[k] = tile[(64 + j) * kFfnLdc + t];
              u1[k] = tile[(65 + j) * kFfnLdc + t];
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int t = tb + 4 * k, r = h0 + t;
              if (t < nh)
                *(__nv_bfloat162 *)(blk + r * 128 + ((((lane >> 2) ^ (r & 7)) << 4) | ((lane & 3) << 2))) =
                    __floats2bfloat162_rn(swiglu_f(g0[k], u0[k]), swiglu_f(g1[k], u1[k]));
            }
          }
        } else {
          // y[row][feature] = tile: lanes walk features, four tokens per step
          float *dst = g.y + (size_t)(inf.b_row + h0) * g.d + inf.mt * 128;
          for (int tb = warp; tb < nh; tb += 16) {
            float v[4][4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
              for (int f4 = 0; f4 < 4; ++f4) v[k][f4] = tile[(32 * f4 + lane) * kFfnLdc + min(tb + 4 * k, nh - 1)];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int t = tb + 4 * k;
              if (t < nh)
#pragma unroll
                for (int f4 = 0; f4 < 4; ++f4) dst[(size_t)t * g.d + 32 * f4 + lane] = v[k][f4];
            }
          }
        }
        epi_sync();  // the tile is free for the next pass
      }
      if (inf.phase == 0) {
        __threadfence();
        asm volatile("fence.proxy.async.global;\n" ::: "memory");
        epi_sync();
        if (threadIdx.x == 0) atomicAdd(g.done + inf.item, 1);  // publish after every thread's stores
      }
      if (threadIdx.x == 0) mbar_arrive(q_empty + q);
    }
  }
  __syncwarp();  // lone-thread roles above: reconverge before the CTA-wide barrier
  tc::fence_before();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                 "r"((uint32_t)(2 * kFfnBN)));
  }
}

int ffn_num_sms() {
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

cudaError_t moe_ffn(const bf16 *x_tiles, int rows, const bf16 *wgu, const bf16 *wd, const int *offs,
                    const int *work, const int *n_work, int max_work, int E, int d, int F, bf16 *act_tiles,
                    float *y, int *err, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (d % 128 || F % 64) return cudaErrorInvalidValue;
  static_assert(FfnSmem::bytes <= 232448, "shared memory of the expert FFN");
  static unsigned long long attr_set = 0;
  int dev = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev >= 64 || !((attr_set >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(moe_ffn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)FfnSmem::bytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set |= 1ull << dev;
  }
  FfnArgs g{};
  g.work = work;
  g.n_work = n_work;
  g.offs = offs;
  g.wgu = wgu;
  g.wd = wd;
  g.x = x_tiles;
  g.done = const_cast<int *>(work) + 2 * max_work;  // zeroed by moe_scatter
  g.next = g.done + max_work;
  g.E = E;
  g.d = d;
  g.F = F;
  g.act = act_tiles;
  g.y = y;
  g.err = err;
  return launch_pdl(moe_ffn_kernel, dim3(ffn_num_sms()), dim3(kFfnThreads), FfnSmem::bytes, st, g);
}

}  // namespace dg
