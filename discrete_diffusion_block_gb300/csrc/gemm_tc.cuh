// Blackwell (sm_103a) tensor-core building blocks: mbarrier waits, TMA
// loads and L2 prefetches, shared-memory matrix descriptors, tcgen05.mma /
// commit / ld, and the split-K GEMM  D[M][N] = A[M][K] . B[N][K]^T  (fp32
// accumulation in tensor memory) used for every projection and expert GEMM
// of the decoder.  The LM head has its own persistent kernel built from the
// same pieces (kernels_lmhead.cu).
//
// Both operands are stored as operand tiles (tiled_index in common.cuh): 128
// rows x 64 columns per tile, already in the 128-byte swizzled order of a
// K-major shared-memory operand, so one contiguous bulk copy stages a tile.
// Roles inside a GEMM CTA (256 threads):
//   warp 0, one thread  -- producer: per 64-wide K step the weight tile (A,
//                          <= 16 KB) and the activation tiles of up to 256
//                          token rows (B) into a 4-stage shared-memory ring;
//                          the first weight tile is requested before the
//                          wait on the previous kernel;
//   warp 1, one thread  -- allocates the TMEM accumulator and issues
//                          tcgen05.mma (M = 128, N <= 256, K = 16) per stage,
//                          releasing each stage with tcgen05.commit;
//   warps 0-7           -- read the accumulator out of TMEM (warp w its
//                          32-lane quarter w % 4, the 32-column chunks of
//                          parity w / 4) and run the fused epilogue.
// Split-K: the SPLIT CTAs of a cluster own 1/SPLIT of K each; after the main
// loop every CTA stores the slices of its fp32 partial tile that its peers
// own to a global exchange buffer (it stays in L2), and CTA j adds the SPLIT
// partials of slice j in rank order (deterministic) and runs the epilogue on
// that slice.
// Every mbarrier wait is bounded; a wait that gives up records an error word
// and lets the CTA finish, so a fault can never hang the GPU.
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace dg {

// Context handed to a GEMM epilogue.
struct TileCtx {
  int m0, n0;      // tile origin in (M, N)
  int m_valid;     // rows of the tile inside M
  int n_valid;     // columns of the tile inside N
  int swz;         // tile layout: element (f, t) at f * ldc + (t ^ (f & swz)); 0 or 31
  int prepared;    // the epilogue's prepare() already staged its inputs in its scratch
};

struct TcArgs {
  int M, N, K;             // D[M][N] = A[M][K] . B[N][K]^T
  const bf16 *a, *b;       // A (weights) and B (activations) as operand tiles (tiled_index)
  int *err;                // device error word (timeouts)
  float *xchg;             // split-K: partial-slice exchange scratch (split_k_xchg_bytes)
};

namespace tc {

constexpr int kBK = 64;                    // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr uint32_t kATileBytes = 128 * 128;
constexpr long long kWaitCycles = 1ll << 31;  // ~1 s at 2 GHz

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(b)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(b)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after ~1 s (or `limit` cycles), records `code` in
// *err and raises the CTA's abort flag, after which every later wait of the
// CTA returns at once.
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity, int *err, int code,
                                         volatile int *abort, long long limit = kWaitCycles) {
  if (*abort) return false;
  const long long t0 = clock64();
  while (!mbar_try_wait(b, parity)) {
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      if (err) atomicExch(err, code);
      *abort = 1;
      return false;
    }
  }
  return true;
}

// Contiguous bulk copy global -> this CTA's shared memory, completion on bar.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];\n" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile with 128-byte swizzling:
// rows of 128 B, 8-row core groups 1024 B apart (stride byte offset), leading
// byte offset unused for this layout, descriptor version 1, swizzle mode 2.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum));
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// The same wait with the loaded registers as in/out operands, so that no use
// of them can be scheduled before it (for code placed between load and wait).
__device__ __forceinline__ void tmem_ld_wait(uint32_t *r) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;\n"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
        "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
        "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}

}  // namespace tc

// ---------------------------------------------------------------------------
// Split-K GEMM for the decoder's skinny products (weights x a few hundred
// tokens).  One CTA owns a 128-row A tile, up to 256 B rows (the MMA N is the
// tile's valid row count rounded up to 16, so a 40-row expert tile costs a
// 128 x 48 MMA) and 1/SPLIT of the K range.  N = 256 keeps the tensor core
// busy per instruction: with N = 64 the single-thread MMA issue and the
// shared-memory operand traffic, not HBM, bounded the mainloop.
//
// The SPLIT CTAs of one output tile form a thread-block cluster.  Each
// stores the slices of its fp32 partial tile that its peers own (W = 256 /
// SPLIT columns per slice) to an exchange buffer in global memory, which
// stays in L2 (measured about three times faster than pushing them through
// distributed shared memory); after a cluster barrier CTA z sums the SPLIT
// partials of slice z in rank order (a fixed order, so results are
// deterministic), its own straight from TMEM, and runs the epilogue on that
// 128 x W slice.  A second cluster barrier ends the unit.
// ---------------------------------------------------------------------------
namespace tc {

__device__ __forceinline__ uint32_t cluster_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_cluster_f4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// Bulk copy of `bytes` from this CTA's shared memory to a peer's (cluster
// addresses dst and bar); completion is signalled on the peer's mbarrier.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
      "r"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::
                   : "memory");
}

constexpr int kSkBN = 256;           // B rows per tile (MMA N upper bound)
constexpr int kSkThreads = 256;      // two warps per TMEM lane quarter in the epilogue
constexpr int kSkStages = 4;
constexpr uint32_t kBChunkBytes = 64 * 128;  // one 64-row B box

// Shared memory of a split-K CTA.  The epilogue area overlays the ring.
// SPLIT > 1: mine = the CTA's reduced output slice [128][W] (element (f, t)
// at f * W + (t ^ (f & 31)), so that the per-row writes and the epilogue's
// column walks are both conflict-free), then the epilogue's scratch.
// SPLIT == 1: red = the tile, [128][kSkBN + 1], then the epilogue scratch.
template <int SPLIT, class Epi>
struct SkSmem {
  static constexpr int W = kSkBN / SPLIT;  // epilogue slice width
  static constexpr uint32_t stage_bytes = kATileBytes + kSkBN * 128;
  static constexpr size_t ring = (size_t)kSkStages * stage_bytes;
  static constexpr uint32_t slice_bytes = 128u * W * 4u;
  static constexpr size_t mine = SPLIT > 1 ? slice_bytes : 0;
  static constexpr int red_ld = kSkBN + 1;  // odd: column walks are conflict-free
  static constexpr size_t red = SPLIT > 1 ? 0 : (size_t)128 * red_ld * 4;
  static constexpr size_t epi = mine + red + Epi::extra_smem;
  // pre: the epilogue inputs its prepare() loads early (split > 1), beside
  // the ring so that they can arrive while the main loop runs.
  static constexpr bool prep = SPLIT > 1 && Epi::prep_bytes(W) > 0;
  static constexpr size_t pre_off = ((ring > epi ? ring : epi) + 127) & ~(size_t)127;
  static constexpr size_t pre_bytes = prep ? Epi::prep_bytes(W) : 0;
  static constexpr size_t bars_off = (pre_off + pre_bytes + 15) & ~(size_t)15;
  static constexpr size_t bytes = bars_off + (2 * kSkStages + 1) * 8 + 16 + 1024;
};

// Global scratch of the split-K exchange for a launch of n_ctas CTAs: each
// CTA's partial slices for the SPLIT CTAs of its cluster (the owner's own
// slot unused), 128 x 256 fp32 per CTA whatever SPLIT is.
inline size_t split_k_xchg_bytes(int n_ctas) { return (size_t)n_ctas * 128 * kSkBN * 4; }

}  // namespace tc

template <int SPLIT, class Epi>
__global__ void __launch_bounds__(tc::kSkThreads, 1)
    tc_gemm_sk_kernel(TcArgs g, Epi epi) {
  using S = tc::SkSmem<SPLIT, Epi>;
  constexpr int STAGES = tc::kSkStages, W = S::W;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *full = (uint64_t *)(base + S::bars_off);
  uint64_t *empty = full + STAGES;
  uint64_t *accb = empty + STAGES;
  uint32_t *tmem_slot = (uint32_t *)(accb + 1);
  volatile int *abort = (volatile int *)(tmem_slot + 1);

  // Output units are (256-column N tile, 128-row M tile) pairs.  Cluster c
  // (the SPLIT CTAs blockIdx.x = c * SPLIT + z, one per K range) takes units
  // c, c + n_clusters, ..., so the grid is sized to the machine and the
  // units spread evenly over it.
  // Every CTA of the launch sees the same cluster size: a launch without the
  // SPLIT-CTA clusters this kernel exchanges partials in returns at once.
  if (cluster_ctas() != (uint32_t)SPLIT) {
    if (threadIdx.x == 0 && g.err) atomicExch(g.err, kShapeErrorBase + 1);
    return;
  }
  const int n_items = ceil_div(g.N, tc::kSkBN);
  const int m_tiles = ceil_div(g.M, 128);
  const int n_units = n_items * m_tiles;
  const int cluster = blockIdx.x / SPLIT, n_clusters = gridDim.x / SPLIT;
  if (cluster >= n_units) return;  // every CTA of a cluster decides alike

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int err_seen = threadIdx.x == 64 ? ld_err_word(g.err) : 0;
  const int z = SPLIT > 1 ? (int)(blockIdx.x % SPLIT) : 0;
  const int KT = g.K / tc::kBK;
  const int kb = (int)((long long)KT * z / SPLIT), ke = (int)((long long)KT * (z + 1) / SPLIT);

  if (threadIdx.x == 0) {
    *abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    tc::mbar_init(accb, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     tc::smem_u32(tmem_slot)),
                 "r"((uint32_t)tc::kSkBN));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  auto a_tile = [&](int s) { return base + (size_t)s * S::stage_bytes; };
  auto b_tile = [&](int s) { return base + (size_t)s * S::stage_bytes + tc::kATileBytes; };

  // One k-tile of a unit: the A tile of M block mt and the B tiles of the
  // (up to two) 128-row blocks of N tile y, each one contiguous bulk copy.
  auto a_bytes = [&](int mt) { return (uint32_t)min(128, g.M - 128 * mt) * 128; };
  auto b_rows = [&](int rb) { return max(0, min(128, g.N - 128 * rb)); };
  auto tx_of = [&](int y, int mt) {
    return a_bytes(mt) + (uint32_t)(b_rows(2 * y) + b_rows(2 * y + 1)) * 128;
  };
  auto load_a = [&](int s, int mt, int kt) {
    tc::bulk_load(a_tile(s), g.a + tiled_index(g.M, g.K, 128 * mt, 64 * kt), a_bytes(mt), full + s);
  };
  auto load_b = [&](int s, int y, int kt) {
    for (int h = 0; h < 2; ++h) {
      const int rb = 2 * y + h, rows = b_rows(rb);
      if (rows > 0)
        tc::bulk_load(b_tile(s) + h * 16384, g.b + tiled_index(g.N, g.K, 128 * rb, 64 * kt), (uint32_t)rows * 128,
                      full + s);
    }
  };
  // Weights never change: the first unit's A tiles are requested before the
  // wait on the kernel that produced B.
  const int pre = min(STAGES, ke - kb);
  if (warp == 0 && lane == 0) {
    const int y0 = cluster / m_tiles, mt0 = cluster - y0 * m_tiles;
    for (int i = 0; i < pre; ++i) {
      tc::mbar_expect_tx(full + i, tx_of(y0, mt0));
      load_a(i, mt0, kb + i);
    }
  }
  // The tile of a unit, and (split > 1) this CTA's slice of it.
  auto unit_ctx = [&](int unit) {
    const int y = unit / m_tiles, mt = unit - y * m_tiles;
    TileCtx c;
    c.m0 = mt * 128;
    c.n0 = y * tc::kSkBN;
    c.swz = 0;
    c.prepared = 0;
    c.m_valid = min(128, g.M - c.m0);
    c.n_valid = max(0, min(tc::kSkBN, g.N - c.n0));
    return c;
  };
  auto slice_ctx = [&](const TileCtx &c) {
    TileCtx sub = c;
    sub.n0 = c.n0 + z * W;
    sub.n_valid = min(W, c.n_valid - z * W);
    sub.swz = 31;
    sub.prepared = S::prep ? 1 : 0;
    return sub;
  };
  // The first unit's epilogue inputs: before the dependency wait when they
  // do not come from earlier kernels, else right after it.
  // (Warps 2-3 only: the producer and MMA threads go straight on.)
  if (S::prep && Epi::kPrepEarly && warp >= 2) {
    const TileCtx sub = slice_ctx(unit_ctx(cluster));
    if (sub.n_valid > 0) epi.prepare(sub, base + S::pre_off, threadIdx.x - 64, tc::kSkThreads - 64);
  }
  pdl_wait();
  pdl_trigger();
  // An earlier timeout: do not wait again.  Loaded at the start by an
  // epilogue thread, off the producer's path (its loops check the flag
  // before every copy).
  if (threadIdx.x == 64 && err_seen) *abort = 1;
  if (S::prep && !Epi::kPrepEarly && warp >= 2) {
    const TileCtx sub = slice_ctx(unit_ctx(cluster));
    if (sub.n_valid > 0) epi.prepare(sub, base + S::pre_off, threadIdx.x - 64, tc::kSkThreads - 64);
  }

  int it = 0;     // ring position: k-tiles issued (producer) / consumed (MMA) so far
  int tiles = 0;  // accumulator phase
  for (int unit = cluster; unit < n_units; unit += n_clusters, ++tiles) {
    const int y = unit / m_tiles, mt = unit - y * m_tiles;
    const TileCtx ctx = unit_ctx(unit);
    const int n_mma = max(16, (ctx.n_valid + 15) & ~15);  // MMA N
    const uint32_t tx_bytes = tx_of(y, mt);

    if (warp == 0 && lane == 0) {
      int issued = it;
      for (int kt = kb; kt < ke; ++kt, ++issued) {
        const int s = issued % STAGES, r = issued / STAGES;
        if (r > 0) tc::mbar_wait(empty + s, (r - 1) & 1, g.err, 1, abort);
        if (*abort) break;
        if (issued >= pre) {  // else this stage's A tile is already on its way
          tc::mbar_expect_tx(full + s, tx_bytes);
          load_a(s, mt, kt);
        }
        load_b(s, y, kt);
      }
      if (*abort) {
        // Drain: wait (bounded) for the last copy issued into each stage.
        for (int i = issued - 1; i >= 0 && i >= issued - STAGES; --i) {
          const long long t0 = clock64();
          while (!tc::mbar_try_wait(full + i % STAGES, (i / STAGES) & 1) &&
                 clock64() - t0 < tc::kWaitCycles) {
          }
        }
      }
    } else if (warp == 1 && lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(128, n_mma);
      for (int kt = kb; kt < ke; ++kt) {
        const int i = it + kt - kb, s = i % STAGES, r = i / STAGES;
        tc::mbar_wait(full + s, r & 1, g.err, 2, abort);
        tc::fence_after();
        const uint64_t adesc = tc::sw128_desc(tc::smem_u32(a_tile(s)));
        const uint64_t bdesc = tc::sw128_desc(tc::smem_u32(b_tile(s)));
#pragma unroll
        for (int kk = 0; kk < tc::kBK / 16; ++kk)
          tc::mma_bf16(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kt > kb || kk) ? 1u : 0u);
        tc::mma_commit(empty + s);
      }
      tc::mma_commit(accb);
    }
    it += ke - kb;
    __syncwarp();

    tc::mbar_wait(accb, tiles & 1, g.err, 3, abort);
    tc::fence_after();
    const int row = (warp & 3) * 32 + lane, hc = warp >> 2;  // TMEM lane; parity of this warp's chunks
    const int nchunks = (ctx.n_valid + 31) >> 5;  // 32-column TMEM chunks holding valid outputs
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    unsigned char *extra = base + S::mine + S::red;
    if (SPLIT == 1) {
      float *red = (float *)base;
#pragma unroll 1
      for (int c = hc; c < nchunks; c += 2) {
        uint32_t v[32];
        tc::tmem_ld32(trow + 32 * c, v);
        tc::tmem_ld_wait(v);
#pragma unroll
        for (int j = 0; j < 32; ++j) red[row * S::red_ld + 32 * c + j] = __uint_as_float(v[j]);
      }
      __syncthreads();
      if (ctx.n_valid > 0) epi(red, S::red_ld, ctx, extra);
    } else {
      // Each CTA stores the partial slices that its peers own to global
      // scratch straight from TMEM (slice j of CTA z at xchg[z][j], stored
      // [W tokens][128 rows]: one coalesced 128-byte store per token and
      // warp).  After a cluster barrier (release / acquire at cluster scope)
      // CTA z reads slice z of every peer from L2 and adds the SPLIT partials
      // in rank order (a fixed order: deterministic), its own straight from
      // TMEM, into shared memory, then runs the epilogue on that 128 x W
      // slice.  A second cluster barrier ends the unit: no peer still reads
      // this CTA's scratch past it.  (Shared-memory pushes between the CTAs
      // of a cluster measured about three times slower than L2.)
      constexpr size_t slice_elems = (size_t)128 * W;
      float *xc = g.xchg + (size_t)(blockIdx.x - z) * SPLIT * slice_elems;  // this cluster's [z][j] slices
      const TileCtx sub = slice_ctx(ctx);
#pragma unroll 1
      for (int c = hc; c < nchunks; c += 2) {
        const int sl = (32 * c) / W, o = 32 * c - sl * W;
        if (sl == z) continue;
        uint32_t v[32];
        tc::tmem_ld32(trow + 32 * c, v);
        tc::tmem_ld_wait(v);
        float *dst = xc + ((size_t)z * SPLIT + sl) * slice_elems + (size_t)o * 128 + row;
#pragma unroll
        for (int j = 0; j < 32; ++j) dst[(size_t)j * 128] = __uint_as_float(v[j]);
      }
      // a later unit's epilogue inputs load while the stores drain
      if (S::prep && unit != cluster && sub.n_valid > 0) epi.prepare(sub, base + S::pre_off, threadIdx.x, tc::kSkThreads);
      tc::cluster_sync();  // every CTA's partials are in L2
      float *mine = (float *)base;
      if (sub.n_valid > 0 && !*abort) {
#pragma unroll 1
        for (int c = hc; c < W / 32; c += 2) {
          if (32 * c >= sub.n_valid) break;
          uint32_t own[32];
          tc::tmem_ld32(trow + z * W + 32 * c, own);
          float pv[SPLIT][32];  // pv[q]: CTA q's partial (q != z), indexed at compile time
#pragma unroll
          for (int q = 0; q < SPLIT; ++q) {
            const float *src = xc + ((size_t)q * SPLIT + z) * slice_elems + (size_t)(32 * c) * 128 + row;
#pragma unroll
            for (int j = 0; j < 32; ++j) pv[q][j] = q == z ? 0.0f : src[(size_t)j * 128];
          }
          tc::tmem_ld_wait(own);
          float *mrow = mine + (size_t)row * W;
          float red[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float acc = z == 0 ? __uint_as_float(own[j]) : pv[0][j];
#pragma unroll
            for (int q = 1; q < SPLIT; ++q)  // rank order
              acc += q == z ? __uint_as_float(own[j]) : pv[q][j];
            red[j] = acc;
          }
          if (Epi::kDirect) {  // the epilogue takes this row's sums as they are
            epi.direct(sub, row, 32 * c, red, S::prep ? base + S::pre_off : nullptr);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) mrow[(32 * c + j) ^ (row & 31)] = red[j];
          }
        }
        if (!Epi::kDirect) {
          __syncthreads();
          epi(mine, W, sub, S::prep ? base + S::pre_off : base + S::mine);
        }
      }
      tc::cluster_sync();
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // the next unit's copies reuse this memory
    // The next unit's MMAs overwrite the accumulator and its copies the
    // shared memory the epilogue used.
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
  }
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                 "r"((uint32_t)tc::kSkBN));
  }
}

// ---- host side ---------------------------------------------------------------

// 2-D bf16 tensor map over a row-major [rows][cols] matrix, box = 64 columns x
// box_rows rows, 128-byte swizzle, zero fill outside the matrix.
cudaError_t make_tmap_bf16(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols,
                           uint32_t box_rows);

// Split-K launch: n_clusters clusters of SPLIT CTAs (grid.x = n_clusters *
// SPLIT, cluster dims (SPLIT, 1, 1)); the clusters walk the output units.
template <int SPLIT, class Epi>
cudaError_t launch_tc_sk(const TcArgs &g, const Epi &epi, int n_clusters, cudaStream_t st) {
  using S = tc::SkSmem<SPLIT, Epi>;
  static_assert(S::bytes <= 232448, "shared memory of the split-K GEMM");
  auto kern = tc_gemm_sk_kernel<SPLIT, Epi>;
  static unsigned long long attr_set = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !((attr_set >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::bytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set |= 1ull << dev;
  }
  if (g.K % tc::kBK || g.K / tc::kBK < SPLIT) return cudaErrorInvalidValue;
  if (SPLIT > 1 && !g.xchg) return cudaErrorInvalidValue;
  if (n_clusters <= 0 || g.M <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_clusters * SPLIT, 1, 1);
  cfg.blockDim = dim3(tc::kSkThreads, 1, 1);
  cfg.dynamicSmemBytes = S::bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (SPLIT > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = SPLIT;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, g, epi);
}

}  // namespace dg
