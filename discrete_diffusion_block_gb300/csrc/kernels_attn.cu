// Canvas / context attention over the paged bf16 KV cache.
//
// Mask (DiffusionGemma report §1 and §4; blog "Once Written, a Prefix
// Becomes History"): every query sees every cached prefix key; inside the
// new block of tokens the canvas is bidirectional (denoising) or causal
// (context encoding and the KV-append forward).  Grouped-query attention:
// the G = Hq/Hkv query heads that share KV head g are packed as rows
// (token t, head h) -> row t*G + (h - g*G), so each K/V tile is read once per
// block for all of them.  Long key ranges are split across blocks and the
// partial softmax states combined afterwards (split-KV).
//
// KV pool layout: a (page, KV head) block of page_size keys is stored as
// hd/64 sub-blocks [page_size][64] in the tensor core's 128-byte swizzled
// operand order (16-byte chunk c of slot s at chunk position c ^ (s % 8)), so
// a 64- or 128-key K or V operand tile is one contiguous bulk copy.
//
// The kernel is a tcgen05 tensor-core kernel with one pass over the block's
// key range and an online softmax: per 128-key tile, S = Q K^T (TMEM), the
// tile's raw-score maximum, P = 2^(S*scale - m) as bf16 into tensor memory,
// row sum l in fp32, O += P V (TMEM).  The running maximum m is raised lazily:
// only a row whose maximum grows by more than 2^8 moves to the new reference
// and rescales its accumulator row in TMEM (read, scale, write back) after the
// previous tile's P V has landed; below that P stays <= 2^8 and the final
// O / l does not depend on which reference was used.  Roles (384 threads):
// warp 0 streams Q once (TMA through a 4-D map that packs the G heads of a
// token as consecutive rows) and the K tiles through a three-slot ring; warp
// 6 streams the V tiles through their own three-slot ring (both as bulk
// copies of the pool's pre-swizzled pages, from a page list resolved before
// the dependency wait); warp 1 issues the S = Q K^T MMAs and warp 11 the
// P V MMAs, each from its own thread, so that S of the next tiles never waits
// behind this tile's softmax; two S accumulators and two P tiles let the
// softmax of one tile overlap the tensor work of the next (P is written to
// tensor memory by the softmax threads and read from there as the A operand
// of P V; V is the N-contiguous "MN-major" B operand); warps 2-5 and 7-10 do the softmax, two
// warps per TMEM lane quarter (thread = query row), each on half of a tile's
// keys, exchanging their halves' maxima per tile.  With the key range split
// over several blocks, the blocks of one query tile form a
// cluster: each stages its unnormalised output rows (bf16) and their softmax
// state (m, l) in its own shared memory, and after a cluster barrier each
// block reads the partials of the rows it owns from every block's shared
// memory (distributed shared-memory loads), merges them (weights
// 2^(m_s - m*)) and writes them; no device scratch is used.
#include <cuda.h>

#include <cudaTypedefs.h>

#include <mutex>
#include <unordered_map>

#include "gemm_tc.cuh"
#include "internal.h"

namespace dg {

namespace {

constexpr int kRowsPerBlock = 128;  // query rows (token, head) per block: the MMA M
constexpr int kKeysPerTile = 128;   // keys per S tile: the MMA N of Q K^T, the K of P V

struct AttnParams {
  const bf16 *q;
  const bf16 *k_pool, *v_pool;
  const int *page_table;
  int n_prefix, n_new, Hq, Hkv, G, pg, causal;
  float scale_log2;
  int keys_per_split;
  bf16 *out;       // unsplit launches: the output
  int *err;        // device error words, may be null: [0] a bounded wait gave up, [1] a bad page index
  int n_pages;     // physical pages of the pools, 0 when unknown
  bf16 *final_out; // split launches: where the cluster's merge writes the output
  int out_tiles;   // outputs as operand tiles over [n_req n_new][Hq hd] (the o-projection operand)
  // several requests (blockIdx.z = request * splits + split): request b's
  // n_new rows follow b * n_new rows of q / out, its keys start after
  // req_prefix[b] cached ones, its pages at page_table[b * pages_per_req ...]
  int n_req, splits, pages_per_req;
  int req_prefix[kMaxRequests];
  int req_kps[kMaxRequests];  // keys per split of each request (its own plan; trailing splits empty)
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *(uint32_t *)&v;
}


constexpr int kAttnThreads = 384;  // warps 0, 6: copies; 1, 11: MMAs; 2-5 and 7-10: softmax
constexpr int kAttnPvWarp = 11;
constexpr int kAttnPages = 64;  // 64-key halves whose physical page is looked up before the key loop
constexpr int kAttnSlotHalfBytes = 64 * 128;  // 64 keys x 64 hd bf16 (one 8 KB copy)

// Shared memory (bytes from a 1024-aligned base): Q [HB][128 rows][64]; a
// 3-slot K ring and a 3-slot V ring of 128-key tiles [HB][128 keys][64] (the
// P tiles live in tensor memory, which leaves room for the third slots: the
// key loop is bound by copy latency times ring depth); the page list;
// barriers.  After the key loop the K ring holds the bf16 output rows
// [128][HD] on their way out (unnormalised partial rows of a split block);
// with split keys the V ring holds the rows' softmax states and the merge
// weights (first 8 KB), and the owners of the rows read the peers' staged
// rows and states from the peers' shared memory.
template <int HD>
struct AttnSmem {
  static constexpr int HB = HD / 64;                       // 64-wide hd blocks
  static constexpr int kK = 3, kV = 3;                     // ring depths
  static constexpr size_t tile = (size_t)HB * 16384;       // one 128-key K or V tile, or Q
  static constexpr size_t q = 0;
  static constexpr size_t kring = q + tile;
  static constexpr size_t vring = kring + kK * tile;
  static constexpr size_t pages = vring + kV * tile;       // physical page per 64-key half (ints)
  static constexpr size_t xch = pages + kAttnPages * 4;    // [2 halves][128 rows] fp32: the softmax pairs' exchange
  static constexpr size_t bars = xch + 2 * 128 * 4;
  // q_full, k_full[3], k_empty[3], v_full[3], v_empty[3], s_full[2], s_empty[2], p_full, p_empty[2], o_full
  static constexpr int n_bars = 1 + 2 * kK + 2 * kV + 4 + 4;
  static constexpr size_t bytes = bars + n_bars * 8 + 16 + 1024;
  static_assert((size_t)128 * HD * 2 <= kK * tile, "output staging fits the K ring");
};

// One 64-key half of a K or V operand tile, all zero (keys past the end).
__device__ __align__(128) unsigned char g_zero_half[kAttnSlotHalfBytes];

__device__ __forceinline__ uint4 ld_cluster_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ float2 ld_cluster_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void attn_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(b)) : "memory");
}

// Shared-memory descriptor of the N-contiguous V tile: 8-key groups 1024 B
// apart along K (SBO), 64-wide hd blocks 16 KB apart along N (LBO), 128-byte
// swizzle.
__device__ __forceinline__ uint64_t mn_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16384 >> 4) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// O += P V with P (bf16, two keys per 32-bit column, row = lane) read from
// tensor memory as the A operand.
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accum));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Rows whose running maximum grows by more than this (log2 units) rescale
// their accumulated output; otherwise P = 2^(s - m) stays <= 2^8 and the
// stale maximum is kept (the final O / l does not depend on m).
constexpr float kRescaleLog2 = 8.0f;

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tq, AttnParams p) {
  using S = AttnSmem<HD>;
  constexpr int HB = S::HB, KK = S::kK, KV = S::kV;
  constexpr uint32_t kTileBytes = (uint32_t)S::tile;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *q_full = (uint64_t *)(base + S::bars);
  uint64_t *k_full = q_full + 1, *k_empty = k_full + KK;
  uint64_t *v_full = k_empty + KK, *v_empty = v_full + KV;
  uint64_t *s_full = v_empty + KV, *s_empty = s_full + 2;
  uint64_t *p_full = s_empty + 2, *p_empty = p_full + 1, *o_full = p_empty + 2;
  uint32_t *tmem_slot = (uint32_t *)(o_full + 1);
  volatile int *abort = (volatile int *)(tmem_slot + 1);
  int *pages = (int *)(base + S::pages);
  auto k_tile = [&](int slot) { return base + S::kring + (size_t)slot * S::tile; };
  auto v_tile = [&](int slot) { return base + S::vring + (size_t)slot * S::tile; };

  // Split blocks merge through distributed shared memory: a launch without
  // the splits-CTA clusters returns at once (every block sees the same size).
  if (p.splits > 1 && cluster_ctas() != (uint32_t)p.splits) {
    if (threadIdx.x == 0 && p.err) atomicExch(p.err, kShapeErrorBase + 2);
    return;
  }
  const int g = blockIdx.y, b_req = blockIdx.z / p.splits, split = blockIdx.z - b_req * p.splits;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_total = p.G * p.n_new;
  const int r_cta = blockIdx.x * 128;
  const int n_prefix = p.n_req > 1 ? p.req_prefix[b_req] : p.n_prefix;
  const int *page_table = p.page_table + (size_t)b_req * p.pages_per_req;
  const int tok0 = b_req * p.n_new;  // the request's first row of q and out
  const int n_keys = n_prefix + p.n_new;
  const int kps = p.n_req > 1 ? p.req_kps[b_req] : p.keys_per_split;
  const int k_begin = split * kps;
  int k_end = min(n_keys, k_begin + kps);
  if (p.causal) {
    const int t_max = min(p.n_new - 1, (r_cta + 127) / p.G);
    k_end = min(k_end, n_prefix + t_max + 1);
  }
  const int n_kt = k_end > k_begin ? ceil_div(k_end - k_begin, 128) : 0;

  const int err_seen = threadIdx.x == 0 ? ld_err_word(p.err) : 0;
  if (threadIdx.x == 0) {
    *abort = 0;
    tc::mbar_init(q_full, 1);
    for (int i = 0; i < KK; ++i) {
      tc::mbar_init(k_full + i, 1);
      tc::mbar_init(k_empty + i, 1);
    }
    for (int i = 0; i < KV; ++i) {
      tc::mbar_init(v_full + i, 1);
      tc::mbar_init(v_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(s_full + i, 1);
      tc::mbar_init(s_empty + i, 8);  // one arrival per softmax warp
    }
    tc::mbar_init(p_full, 8);
    tc::mbar_init(p_empty, 1);
    tc::mbar_init(p_empty + 1, 1);
    tc::mbar_init(o_full, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     tc::smem_u32(tmem_slot)),
                 "r"(512u));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  // Physical page of every 64-key half of the block's range (-1 past the
  // last key or on a bad index), before the wait on the previous kernel: the
  // page table was written before it started.  (Requesting those pages' K
  // and V into L2 here as well delayed the first K tile: the prefetches go
  // through the same bulk-copy path as the ring's loads.)
  const int n_halves = 2 * n_kt;
  if (warp == 0) {
    for (int i = lane; i < n_halves; i += 32) {
      const int key = k_begin + 64 * i;
      int pg_i = key < k_end ? page_table[key / p.pg] : -1;
      if (pg_i >= 0 && p.n_pages > 0 && pg_i >= p.n_pages) {
        if (p.err) atomicExch(p.err + 1, 39);  // reported, not an abort: later blocks still run
        pg_i = -1;
      }
      if (i < kAttnPages) pages[i] = pg_i;
    }
  }
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0 && err_seen) *abort = 1;
  __syncwarp();  // lone-thread roles above: reconverge before the CTA-wide barrier
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  // S double buffer: columns [0,128) [128,256); O: [256, 256+HD); P double
  // buffer (bf16 pairs): [384, 448) [448, 512)
  const uint32_t t_s = tmem, t_o = tmem + 256, t_p = tmem + 384;

  // One 128-key K or V tile: per 64-key half, the page's hd sub-blocks; two
  // halves of one page that follow each other move as one copy; a half past
  // the block's last key (or on a bad page index) is a zero half (its P is
  // zero; V must hold finite values).
  auto load_tile = [&](const bf16 *pool, unsigned char *dst, int kt, uint64_t *bar) {
    const int key0 = k_begin + 128 * kt;
    int pgs[2];
    for (int h = 0; h < 2; ++h) {
      const int key = key0 + 64 * h, hi = 2 * kt + h;
      int pg_i;
      if (hi < kAttnPages) {
        pg_i = pages[hi];
      } else {
        pg_i = key < k_end ? page_table[key / p.pg] : -1;
        if (pg_i >= 0 && p.n_pages > 0 && pg_i >= p.n_pages) pg_i = -1;
      }
      pgs[h] = pg_i;
    }
    const bool whole = pgs[0] >= 0 && pgs[1] == pgs[0] && (key0 % p.pg) + 128 <= p.pg;
    tc::mbar_expect_tx(bar, kTileBytes);
    for (int h = 0; h < (whole ? 1 : 2); ++h) {
      const uint32_t bytes = whole ? 2 * kAttnSlotHalfBytes : kAttnSlotHalfBytes;
      const size_t off = pgs[h] < 0 ? 0 : ((size_t)pgs[h] * p.Hkv + g) * p.pg * HD + (size_t)((key0 + 64 * h) % p.pg) * 64;
      for (int b = 0; b < HB; ++b)
        tc::bulk_load(dst + (size_t)b * 16384 + h * kAttnSlotHalfBytes,
                  pgs[h] < 0 ? (const void *)g_zero_half : (const void *)(pool + off + (size_t)b * p.pg * 64), bytes, bar);
    }
  };
  // Bounded wait for the last copy into each of `depth` slots (after an abort).
  auto drain = [&](uint64_t *full, int issued, int depth) {
    for (int i = issued - 1; i >= 0 && i >= issued - depth; --i) {
      const long long t0 = clock64();
      while (!tc::mbar_try_wait(full + i % depth, (i / depth) & 1) && clock64() - t0 < tc::kWaitCycles) {
      }
    }
  };

  if (warp == 0) {  // Q, then the K ring (S of a tile needs only its K)
    if (lane == 0 && n_kt > 0) {
      tc::mbar_expect_tx(q_full, (uint32_t)(HB * 16384));
      for (int b = 0; b < HB; ++b) {
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes "
            "[%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(tc::smem_u32(base + S::q + (size_t)b * 16384)),
            "l"((uint64_t)&tq), "r"(64 * b), "r"(0), "r"(g), "r"(tok0 + r_cta / p.G), "r"(tc::smem_u32(q_full))
            : "memory");
      }
      int nk = 0;
      for (; nk < n_kt; ++nk) {
        const int slot = nk % KK;
        if (nk >= KK) tc::mbar_wait(k_empty + slot, ((nk / KK) - 1) & 1, p.err, 31, abort);
        if (*abort) break;
        load_tile(p.k_pool, k_tile(slot), nk, k_full + slot);
      }
      if (*abort) drain(k_full, nk, KK);
    }
  } else if (warp == 6) {  // the V ring
    if (lane == 0 && n_kt > 0) {
      int nv = 0;
      for (; nv < n_kt; ++nv) {
        const int slot = nv % KV;
        if (nv >= KV) tc::mbar_wait(v_empty + slot, ((nv / KV) - 1) & 1, p.err, 30, abort);
        if (*abort) break;
        load_tile(p.v_pool, v_tile(slot), nv, v_full + slot);
      }
      if (*abort) drain(v_full, nv, KV);
    }
  } else if (warp == 1) {
    if (lane == 0 && n_kt > 0) {
      const uint32_t idesc_s = tc::idesc_bf16(128, 128);
      tc::mbar_wait(q_full, 0, p.err, 32, abort);
      auto issue_s = [&](int i) {  // S[i & 1] = Q K_i^T
        const int slot = i % KK, buf = i & 1;
        if (i >= 2) tc::mbar_wait(s_empty + buf, ((i >> 1) - 1) & 1, p.err, 33, abort);
        tc::mbar_wait(k_full + slot, (i / KK) & 1, p.err, 34, abort);
        tc::fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint64_t adesc = tc::sw128_desc(tc::smem_u32(base + S::q + (size_t)(kk >> 2) * 16384)) + 2 * (kk & 3);
          const uint64_t bdesc = tc::sw128_desc(tc::smem_u32(k_tile(slot) + (size_t)(kk >> 2) * 16384)) + 2 * (kk & 3);
          tc::mma_bf16(t_s + buf * 128, adesc, bdesc, idesc_s, kk ? 1u : 0u);
        }
        tc::mma_commit(s_full + buf);
        tc::mma_commit(k_empty + slot);
      };
      for (int i = 0; i < n_kt; ++i) issue_s(i);
    }
  } else if (warp == kAttnPvWarp) {
    // P V of every tile, from its own thread: issuing S of the next tiles
    // does not wait for this tile's softmax (each thread's commits track the
    // MMAs it issued).
    if (lane == 0 && n_kt > 0) {
      const uint32_t idesc_o = tc::idesc_bf16(128, HD) | (1u << 16);  // B (V) N-contiguous
      for (int i = 0; i < n_kt; ++i) {
        const int slot = i % KV;
        tc::mbar_wait(p_full, i & 1, p.err, 35, abort);
        tc::mbar_wait(v_full + slot, (i / KV) & 1, p.err, 29, abort);
        tc::fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // 128 keys, 16 (8 columns of P) per MMA
          const uint64_t bdesc = mn_desc(tc::smem_u32(v_tile(slot))) + (uint64_t)kk * (2048 >> 4);
          mma_bf16_tmem_a(t_o, t_p + 64 * (i & 1) + 8 * kk, bdesc, idesc_o, (i | kk) ? 1u : 0u);
        }
        tc::mma_commit(p_empty + (i & 1));
        tc::mma_commit(v_empty + slot);
      }
      tc::mma_commit(o_full);
    }
  } else {
    // ---- softmax warps: two per TMEM lane quarter (warps 2-5: keys 0-63 of a
    // tile, warps 7-10: keys 64-127); thread = query row; the pair exchanges
    // its halves' maxima through shared memory (named barrier 1 + quarter)
    const int half = warp >= 7 ? 1 : 0;
    const int q4 = warp & 3, row = 32 * q4 + lane, r = r_cta + row;
    const bool ok = r < rows_total;
    const int lim = p.causal ? n_prefix + (ok ? r / p.G : 0) : n_keys - 1;
    const int last = min(k_end - 1, lim);  // last key this row sees in the block's range
    const float NEG = __int_as_float(0xff800000);
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    float *xch = (float *)(base + S::xch);  // [2 halves][128 rows]
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;\n" ::"r"(1 + q4) : "memory"); };
    float m = NEG, l = 0.0f;  // l: this half's share of the row sum
    for (int i = 0; i < n_kt; ++i) {
      const int buf = i & 1;
      tc::mbar_wait(s_full + buf, (i >> 1) & 1, p.err, 36, abort);
      tc::fence_after();
      const int key_base = k_begin + 128 * i + 64 * half;
      uint32_t x[2][32];
#pragma unroll
      for (int c = 0; c < 2; ++c) tc::tmem_ld32(t_s + buf * 128 + lane_off + 64 * half + 32 * c, x[c]);
#pragma unroll
      for (int c = 0; c < 2; ++c) tc::tmem_ld_wait(x[c]);  // ties every loaded register to the wait
      tc::fence_before();
      __syncwarp();
      if (lane == 0) attn_arrive(s_empty + buf);
      // keys this row must not see are -inf (only in a half that holds some)
      const int nvalid = min(64, last - key_base + 1);  // <= 0: none
      if (nvalid < 64) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (32 * c + j >= nvalid) x[c][j] = 0xff800000u;
      }
      // maximum of the raw scores of this half (the scale is positive), four
      // chains, then the pair's maximum
      float a0 = __int_as_float(0xff800000), a1 = a0, a2 = a0, a3 = a0;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          a0 = fmaxf(a0, __uint_as_float(x[c][j]));
          a1 = fmaxf(a1, __uint_as_float(x[c][j + 1]));
          a2 = fmaxf(a2, __uint_as_float(x[c][j + 2]));
          a3 = fmaxf(a3, __uint_as_float(x[c][j + 3]));
        }
      const float hmax = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
      xch[half * 128 + row] = hmax;
      pair_sync();
      const float tmax = fmaxf(hmax, xch[(half ^ 1) * 128 + row]) * p.scale_log2;
      pair_sync();  // both read before the next tile's maxima overwrite the slots
      const float m_new = fmaxf(m, tmax);
      const bool grow = m_new > m + kRescaleLog2;  // false while both are -inf; the same in both halves
      // P tile i & 1 is free once P V of tile i - 2 is done
      if (i >= 2) tc::mbar_wait(p_empty + (i & 1), ((i >> 1) - 1) & 1, p.err, 37, abort);
      const float m_old = m;
      if (grow) m = m_new;
      // P = 2^(x scale - m): one FMA and one ex2 per key; -inf keys give 0.
      // Each 32-key group goes to the row's P columns in tensor memory as
      // soon as it is packed (this half: columns 32 half .. 32 half + 31).
      const float nmu = m == NEG ? 0.0f : -m;
      float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
      const uint32_t prow = t_p + 64 * (i & 1) + 32 * half + lane_off;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float p0 = ex2(fmaf(__uint_as_float(x[c][j]), p.scale_log2, nmu));
          const float p1 = ex2(fmaf(__uint_as_float(x[c][j + 1]), p.scale_log2, nmu));
          if ((j & 6) == 0) s0 += p0 + p1;
          else if ((j & 6) == 2) s1 += p0 + p1;
          else if ((j & 6) == 4) s2 += p0 + p1;
          else s3 += p0 + p1;
          pk[j >> 1] = pack_bf16(p0, p1);
        }
        tmem_st16(prow + 16 * c, pk);
      }
      // rows whose maximum grew: O (and l) to the new reference, O <- O 2^(m_old - m);
      // each half rescales its half of the O columns
      float f = 1.0f;
      if (__any_sync(0xffffffffu, grow) && i > 0) {
        // O must hold P V of every earlier tile: wait for tile i - 1's
        tc::mbar_wait(p_empty + ((i - 1) & 1), ((i - 1) >> 1) & 1, p.err, 40, abort);
        tc::fence_after();
        f = grow ? ex2(m_old - m) : 1.0f;  // m_old = -inf: 0 (O holds zeros)
#pragma unroll 1
        for (int c = half * (HD / 64); c < (half + 1) * (HD / 64); ++c) {
          uint32_t o[32];
          tc::tmem_ld32(t_o + lane_off + 32 * c, o);
          tc::tmem_ld_wait(o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
          tmem_st32(t_o + lane_off + 32 * c, o);
        }
      }
      l = l * f + ((s0 + s1) + (s2 + s3));
      asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");  // P (and O) written before the release
      tc::fence_before();
      __syncwarp();
      if (lane == 0) attn_arrive(p_full);
    }
    // the row sum of both halves
    xch[half * 128 + row] = l;
    pair_sync();
    const float lt = half ? xch[row] + l : l + xch[128 + row];  // keys 0-63 first
    // ---- output: TMEM -> shared rows -> coalesced stores --------------------
    if (n_kt > 0) {
      tc::mbar_wait(o_full, 0, p.err, 38, abort);
      tc::fence_after();
    }
    const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
    uint4 *orow = (uint4 *)(base + S::kring) + (size_t)row * (HD / 8);  // the K ring is idle now
#pragma unroll 1
    for (int c = half * (HD / 64); c < (half + 1) * (HD / 64); ++c) {
      uint32_t v[32];
      if (n_kt > 0) {
        tc::tmem_ld32(t_o + lane_off + 32 * c, v);
        tc::tmem_ld_wait(v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0u;
      }
      const float sc = p.out ? inv : 1.0f;  // split blocks keep the unnormalised sum
#pragma unroll
      for (int j = 0; j < 32; j += 8) {  // bf16 chunk of 8 columns, slot rotated by row: conflict-free
        const int q = ((32 * c + j) >> 3) ^ (row & 7);
        uint4 w;
        w.x = pack_bf16(__uint_as_float(v[j]) * sc, __uint_as_float(v[j + 1]) * sc);
        w.y = pack_bf16(__uint_as_float(v[j + 2]) * sc, __uint_as_float(v[j + 3]) * sc);
        w.z = pack_bf16(__uint_as_float(v[j + 4]) * sc, __uint_as_float(v[j + 5]) * sc);
        w.w = pack_bf16(__uint_as_float(v[j + 6]) * sc, __uint_as_float(v[j + 7]) * sc);
        orow[q] = w;
      }
    }
    if (!p.out && half == 0) ((float2 *)(base + S::vring))[row] = make_float2(m, lt);  // split blocks: the row's softmax state
  }
  __syncwarp();  // lone-thread roles above: reconverge before the CTA-wide barrier
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(512u));
  }
  if (p.out) {
    // Rows out of shared memory, one warp per row, lanes along hd.
    const uint4 *stage = (const uint4 *)(base + S::kring);
    for (int rr = warp; rr < 128; rr += kAttnThreads / 32) {
      const int r = r_cta + rr;
      if (r >= rows_total) break;
      const int t = tok0 + r / p.G, h = g * p.G + r % p.G;
      for (int c8 = lane; c8 < HD / 8; c8 += 32)
        *(uint4 *)(p.out + (p.out_tiles ? tiled_index(p.n_req * p.n_new, p.Hq * HD, t, h * HD + 8 * c8)
                                        : ((size_t)t * p.Hq + h) * HD + 8 * c8)) = stage[(size_t)rr * (HD / 8) + (c8 ^ (rr & 7))];
    }
    return;
  }
  // Split-KV merge inside the cluster of this query tile's blocks.  Block z
  // owns rows [z n, z n + n), n = ceil(128 / NS).  After a cluster barrier
  // (every block has staged its unnormalised output rows and their softmax
  // states) the owner reads the NS partials of its rows straight from the
  // blocks' shared memory (distributed shared-memory loads, all of a column's
  // in flight) and merges them with weights 2^(m_s - m*); a second barrier
  // keeps each block's staged rows until its peers have read them.
  const int NS = p.splits;
  const int n_own = (128 + NS - 1) / NS;
  const uint32_t stage_sa = tc::smem_u32(base + S::kring), ml_sa = tc::smem_u32(base + S::vring);
  __syncwarp();
  tc::cluster_sync();  // every block staged its rows and states
  const int z = split, r0 = z * n_own, n_mine = max(0, min(128, r0 + n_own) - r0);
  // Once per owned row: the partials' weights 2^(m_s - m*) (0 for a split
  // that saw no key), 1 / L and the output row (token, head), into the V ring
  // past the staged softmax states; then every thread merges float4 columns
  // with them.
  const float NEG = __int_as_float(0xff800000);
  float *wtab = (float *)(base + S::vring + 2048);  // [n_own][8] weights, then [n_own] 1 / L
  int *otab = (int *)(wtab + 9 * n_own);            // [n_own] (token << 12) | head, -1 past the rows
  for (int lr = threadIdx.x; lr < n_mine; lr += kAttnThreads) {
    const int rr = r0 + lr, r = r_cta + rr;
    float2 ml[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      ml[q] = q < NS ? ld_cluster_f2(tc::cluster_addr(ml_sa + 8u * (uint32_t)rr, (uint32_t)q)) : make_float2(NEG, 0.0f);
    float mx = NEG;
#pragma unroll
    for (int q = 0; q < 8; ++q) mx = fmaxf(mx, ml[q].x);
    float L = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float w = 0.0f;
      if (q < NS && ml[q].x != NEG) {
        w = ex2(ml[q].x - mx);
        L += w * ml[q].y;
      }
      wtab[lr * 8 + q] = w;
    }
    wtab[8 * n_own + lr] = L > 0.0f ? 1.0f / L : 0.0f;
    otab[lr] = r < rows_total ? ((tok0 + r / p.G) << 12) | (g * p.G + r % p.G) : -1;
  }
  __syncthreads();
  // Two 8-column chunks per thread at a time, the loads of both in flight
  // before the sums; partials summed in split order.
  const int n_items = n_mine * (HD / 8);
  for (int i0 = threadIdx.x; i0 < n_items; i0 += 2 * kAttnThreads) {
    float w[2][8];
    uint4 o[2][8];
    int th[2], c8s[2], lrs[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int idx = i0 + u * kAttnThreads;
      th[u] = -1;
      if (idx >= n_items) continue;
      const int lr = idx / (HD / 8), c8 = idx - lr * (HD / 8), rr = r0 + lr;
      th[u] = otab[lr];
      c8s[u] = c8;
      lrs[u] = lr;
      // the staging order travels with the rows: chunk c8 of row rr sits at slot c8 ^ (rr & 7)
      const uint32_t off = stage_sa + 16u * (uint32_t)(rr * (HD / 8) + (c8 ^ (rr & 7)));
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        w[u][q] = (q < NS && th[u] >= 0) ? wtab[lr * 8 + q] : 0.0f;
        if (w[u][q] != 0.0f) o[u][q] = ld_cluster_u4(tc::cluster_addr(off, (uint32_t)q));
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (th[u] < 0) continue;
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (w[u][q] == 0.0f) continue;
        const uint32_t wd[4] = {o[u][q].x, o[u][q].y, o[u][q].z, o[u][q].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[2 * e] += w[u][q] * __uint_as_float(wd[e] << 16);
          acc[2 * e + 1] += w[u][q] * __uint_as_float(wd[e] & 0xffff0000u);
        }
      }
      const float invL = wtab[8 * n_own + lrs[u]];
      const int t = th[u] >> 12, h = th[u] & 4095, c8 = c8s[u];
      uint4 v;
      v.x = pack_bf16(acc[0] * invL, acc[1] * invL);
      v.y = pack_bf16(acc[2] * invL, acc[3] * invL);
      v.z = pack_bf16(acc[4] * invL, acc[5] * invL);
      v.w = pack_bf16(acc[6] * invL, acc[7] * invL);
      *(uint4 *)(p.final_out + (p.out_tiles ? tiled_index(p.n_req * p.n_new, p.Hq * HD, t, h * HD + 8 * c8)
                                            : ((size_t)t * p.Hq + h) * HD + 8 * c8)) = v;
    }
  }
  __syncwarp();
  tc::cluster_sync();  // the peers have read this block's staged rows and states
}

struct SplitPlan {
  int splits, keys_per_split;
};

// Key splits of one request with n_prefix cached keys (a batch of requests
// uses each request's own plan, so that its results do not depend on the
// others': the batch's grid has the largest split count, and a request's
// splits past its own are empty).
SplitPlan plan_splits(const AttnShape &s, int n_prefix) {
  const int G = s.Hq / s.Hkv;
  const int base = s.Hkv * ceil_div(G * s.n_new, kRowsPerBlock);
  const int n_keys = n_prefix + s.n_new;
  const int n_kb = ceil_div(n_keys, kKeysPerTile);
  int splits = 148 / base;  // about one wave: one 192 KB block per SM
  if (splits > 8) splits = 8;  // the blocks of a query tile form one (portable) cluster
  if (splits > n_kb) splits = n_kb;
  if (splits < 1) splits = 1;
  const int kps = ceil_div(n_kb, splits) * kKeysPerTile;
  SplitPlan pl;
  pl.keys_per_split = kps;
  pl.splits = ceil_div(n_keys, kps);
  if (pl.splits < 1) pl.splits = 1;
  return pl;
}

}  // namespace

int attention_launch_count(const AttnShape &s) { return s.n_new <= 0 ? 0 : 1; }

// The split-KV partial states never leave the chip (the blocks of a query
// tile merge them through distributed shared memory): no device scratch.
size_t attention_workspace_bytes(const AttnShape &) { return 0; }

namespace {

// Tensor maps of the attention operands (encoded once per address and shape).
PFN_cuTensorMapEncodeTiled_v12000 attn_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    cudaGetLastError();
  }
  return fn;
}

struct AttnMapKey {
  const void *ptr;
  uint64_t d0, d1, d2, d3;
  bool operator==(const AttnMapKey &o) const {
    return ptr == o.ptr && d0 == o.d0 && d1 == o.d1 && d2 == o.d2 && d3 == o.d3;
  }
};
struct AttnMapHash {
  size_t operator()(const AttnMapKey &k) const {
    return std::hash<const void *>()(k.ptr) ^ (k.d0 * 0x9e3779b97f4a7c15ull) ^ (k.d1 << 7) ^ (k.d2 << 17) ^ (k.d3 << 29);
  }
};
std::mutex g_attn_mu;
std::unordered_map<AttnMapKey, CUtensorMap, AttnMapHash> g_attn_maps;

// rank-2 ([rows][cols], box 64 x box_rows) or rank-4 ([d3][d2][d1][d0], box
// 64 x G x 1 x 128/G) bf16 map, 128-byte swizzle, zero fill outside.
cudaError_t attn_map(CUtensorMap *map, const void *ptr, int rank, const uint64_t *dims,
                     const uint64_t *strides_bytes, const uint32_t *box) {
  const AttnMapKey key{ptr, dims[0], dims[1], rank > 2 ? dims[2] : 0, rank > 3 ? dims[3] : 0};
  std::lock_guard<std::mutex> lock(g_attn_mu);
  auto it = g_attn_maps.find(key);
  if (it != g_attn_maps.end()) {
    *map = it->second;
    return cudaSuccess;
  }
  auto fn = attn_encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t d[4], st[3];
  cuuint32_t bx[4], es[4] = {1, 1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) st[i] = strides_bytes[i];
  // no L2 promotion: a box never asks for bytes past the rows it names, which
  // matters for pool maps whose row extent is only an upper bound
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr), d, st, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  if (g_attn_maps.size() > 4096) g_attn_maps.clear();
  g_attn_maps.emplace(key, *map);
  return cudaSuccess;
}

template <int HD>
cudaError_t launch_attn(const CUtensorMap &tq, const AttnParams &p, dim3 grid, cudaStream_t st) {
  // the key splits of one request's query tile form a cluster (grid.z = requests x splits)
  using S = AttnSmem<HD>;
  static_assert(S::bytes <= 232448, "shared memory of the attention kernel");
  static unsigned long long attr_set = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !((attr_set >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(attn_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::bytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set |= 1ull << dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kAttnThreads, 1, 1);
  cfg.dynamicSmemBytes = S::bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.splits > 1) {  // the key splits of a query tile: one cluster
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = p.splits;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, attn_tc_kernel<HD>, tq, p);
}

}  // namespace

cudaError_t attention(const bf16 *q, const bf16 *k_pool, const bf16 *v_pool, const int *page_table,
                      const AttnShape &s, bf16 *out, void *ws, size_t ws_bytes, cudaStream_t st,
                      int *err, bool out_tiles) {
  if (s.n_new <= 0) return cudaSuccess;
  if ((s.hd != 64 && s.hd != 128) || s.Hq % s.Hkv != 0 || s.Hq > 4096 || s.n_new >= (1 << 19) || s.pg % 64 != 0)
    return cudaErrorInvalidValue;
  const int G = s.Hq / s.Hkv;
  if (128 % G) return cudaErrorInvalidValue;
  SplitPlan pl = plan_splits(s, s.n_prefix);
  int req_kps[kMaxRequests] = {};
  if (s.n_req > 1) {
    pl.splits = 1;
    for (int b = 0; b < s.n_req; ++b) {
      const SplitPlan pb = plan_splits(s, s.req_prefix[b]);
      req_kps[b] = pb.keys_per_split;
      pl.splits = max(pl.splits, pb.splits);
    }
  }
  AttnParams p;
  p.q = q;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.page_table = page_table;
  p.n_prefix = s.n_prefix;
  p.n_new = s.n_new;
  if (s.n_req < 1 || s.n_req > kMaxRequests) return cudaErrorInvalidValue;
  p.n_req = s.n_req;
  p.splits = pl.splits;
  p.pages_per_req = s.pages_per_req;
  for (int b = 0; b < kMaxRequests; ++b) {
    p.req_prefix[b] = b < s.n_req ? s.req_prefix[b] : 0;
    p.req_kps[b] = req_kps[b];
  }
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.G = G;
  p.pg = s.pg;
  p.causal = s.causal;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)s.hd));
  p.keys_per_split = pl.keys_per_split;
  p.err = err;
  p.n_pages = s.n_pages;
  const int rows_total = G * s.n_new;
  (void)ws;
  (void)ws_bytes;
  p.out = pl.splits > 1 ? nullptr : out;  // split blocks merge in the cluster, then write final_out
  p.final_out = out;
  p.out_tiles = out_tiles ? 1 : 0;
  if (out_tiles && (s.Hq * s.hd) % 64) return cudaErrorInvalidValue;
  // Q [T][Hq][hd] as a 4-D tensor (hd, G, Hkv, T): a box of 64 x G x 1 x 128/G
  // lands as 128 rows (token, head of the group) of 128 bytes.
  CUtensorMap tq;
  {
    const uint64_t dims[4] = {(uint64_t)s.hd, (uint64_t)G, (uint64_t)s.Hkv, (uint64_t)s.n_new * s.n_req};
    const uint64_t strides[3] = {(uint64_t)s.hd * 2, (uint64_t)G * s.hd * 2, (uint64_t)s.Hq * s.hd * 2};
    const uint32_t box[4] = {64, (uint32_t)G, 1, (uint32_t)(128 / G)};
    cudaError_t e = attn_map(&tq, q, 4, dims, strides, box);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(ceil_div(rows_total, kRowsPerBlock), s.Hkv, pl.splits * s.n_req);
  return s.hd == 128 ? launch_attn<128>(tq, p, grid, st) : launch_attn<64>(tq, p, grid, st);
}

}  // namespace dg
