// Routed-expert feed-forward of one MoE layer as a single persistent
// warp-specialised tcgen05 kernel: for every routed expert e with token rows
// X_e (gathered in expert order),
//   act_e = SiLU(X_e Wg_e^T) * (X_e Wu_e^T)        (phase A, "gate/up")
//   y_e   = act_e Wd_e^T                           (phase B, "down")
//
// Units.  A work item is (expert, up to 128 of its rows).  A phase A unit is
// (item, 128 features): two MMAs per k-step, the gate rows into one TMEM
// accumulator and the up rows of the same features into a second one, both
// against the one copy of the item's rows staged for that k-step -- so a
// thread that owns a feature's TMEM lane holds its gate and up projections
// and SwiGLU needs no exchange.  A phase B unit is (item, 256 rows of
// W_down), again two accumulators sharing one staged act tile.  Sharing the
// B operand between two weight blocks halves the re-reads of the item's rows,
// which are as many bytes as the weights themselves.  All units sit in one
// list, phase A first; CTA b (one per SM) starts with unit b and then takes
// the next unit from a global counter.  A phase B unit needs the whole act row block of its item: its
// producer first requests the unit's leading weight tiles, then waits
// (bounded) until the item's phase A units have all published their outputs
// (per-item counter, release/acquire, then a proxy fence before the copies
// read them).
//
// Overflow split.  When the phase A units exceed a whole number of waves by
// at most a quarter of the grid, those last units would run as a nearly
// empty extra wave of full units (a unit's k-steps are latency-bound, ~26 us
// for d = 2816).  Instead each runs as four parts over a quarter of K on
// separate SMs: a part stores its fp32 gate and up sums in a slot and takes
// a ticket; the part whose ticket is last (every other part's sums already
// stored) sums the four slots in part order -- the same bits whichever CTAs
// ran the parts -- and writes and publishes the item's act tile like a
// whole unit.  No part waits for another.
//
// Operands.  Expert weights and the item rows (gathered by moe_scatter, and
// the SwiGLU output written here by phase A) are stored as 16 KB tiles of 128
// rows x 64 columns already in the tensor core's swizzled shared-memory order,
// so each k-step of a unit stages its operands with three contiguous bulk
// copies (two weight tiles, the item's valid rows).
//
// Roles (320 threads):
//   warp 8, one thread  -- takes units, hands them to the other roles through
//                          a 4-deep shared-memory queue, and streams the
//                          operands per k-step into a 4-stage ring (48 KB a
//                          stage);
//   warp 9, one thread  -- owns all 512 TMEM columns and issues tcgen05.mma
//                          (M = 128, N = rows rounded up to 16), unit n into
//                          accumulator pair n & 1;
//   warps 0-7           -- epilogue straight from TMEM: warp w reads lane
//                          quarter w % 4 and token columns 64 (w / 4) ..
//                          64 (w / 4) + 63 of the pair, computes SwiGLU and
//                          writes the act tile (A) or writes bf16 y rows (B)
//                          with coalesced stores, while the tensor core
//                          already works on the next unit.
// Every wait is bounded; a wait that gives up records an error word and makes
// the CTA's later waits return at once.
#include <cuda.h>

#include "gemm_tc.cuh"
#include "internal.h"

namespace dg {

namespace {

constexpr int kFfnStages = 4;
// 128-row blocks of W_down per down unit (two accumulators sharing one
// staged act tile).  Measured: with one block a down unit's k-step took as
// long as with two (the ring's four stages in flight, not the bytes per
// stage, set the pace), so two blocks do twice the work per k-step.
constexpr int kDownBlocks = 2;
constexpr int kFfnEpiWarps = 8;
constexpr int kFfnEpiThreads = 32 * kFfnEpiWarps;
constexpr int kFfnThreads = kFfnEpiThreads + 64;
constexpr int kFfnProducerWarp = kFfnEpiWarps, kFfnMmaWarp = kFfnEpiWarps + 1;
constexpr int kFfnBN = kExpertTileRows;  // rows per item = MMA N upper bound
constexpr int kFfnQueue = 4;
constexpr int kFfnSplitParts = 4;  // K-range parts of a split gate/up unit
constexpr uint32_t kFfnATileBytes = 128 * 128;  // one weight tile, up to 128 rows x 64
constexpr uint32_t kFfnBBytes = kFfnBN * 128;
constexpr uint32_t kFfnStageBytes = 2 * kFfnATileBytes + kFfnBBytes;
constexpr uint32_t kFfnPairCols = 2 * kFfnBN;  // TMEM columns of one accumulator pair

struct UnitInfo {
  int u;        // unit index, -1 = no more units
  int phase;    // 0: gate/up, 1: down
  int item, mt, b_row, n_valid, e;
  int a_rows;   // valid rows of each weight tile (phase A: features in the block)
  int n_acc;    // weight blocks (accumulators) of the unit: 2 (gate, up), or kDownBlocks or fewer (down)
  int kb, ke;   // the unit's k-steps
  int part;     // a split gate/up unit: this part's index (its K range), else -1
  int ov;       // a split gate/up unit: its index among the split units
  int nparts;   // a split gate/up unit: its number of parts
  int pad[2];
};

struct FfnSmem {
  static constexpr size_t ring = (size_t)kFfnStages * kFfnStageBytes;
  static constexpr size_t queue = ring;  // UnitInfo [kFfnQueue]
  static constexpr size_t bars = (queue + kFfnQueue * sizeof(UnitInfo) + 15) & ~(size_t)15;
  // full[S], empty[S], acc_full[2], acc_empty[2], q_full[Q], q_empty[Q]; TMEM address; abort flag
  static constexpr size_t bytes = bars + (2 * kFfnStages + 4 + 2 * kFfnQueue) * 8 + 16 + 1024;
};

// Operands are stored as 16 KB tiles (128 rows x 64 columns, in the
// tensor core's 128-byte swizzled shared-memory order); one contiguous bulk
// copy moves a weight tile, one moves the valid rows of an item's tile.
struct FfnArgs {
  const int *work, *n_work, *offs;
  const bf16 *wgu;  // per expert: operand tiles of W_gate [F][d], then of W_up [F][d]
  const bf16 *wd;   // per expert: operand tiles of W_down [d][F]
  const bf16 *x;    // [item][d/64] tiles: the item's token rows (fp8: [item][d/128] e4m3 tiles)
  // fp8 != 0: the gate/up products take e4m3 operands: wgu8 holds W_gate /
  // W_up as e4m3 operand tiles (same order as wgu), kw their rows' scale
  // exponents [E][2][F], kx the exponents of the token rows [rows]
  int fp8;
  const uint8_t *wgu8;
  const int *kw, *kx;
  int *done;   // [max_work] phase A units finished per item
  int *next;   // unit counter
  // Split gate/up units (the overflow past a whole number of waves): each
  // part stores its sums in a slot of part_buf ([2 (gate, up)][32 groups of
  // 4 token columns][128 features][4] fp32) and takes a ticket from
  // part_cnt[unit]; the last part sums the parts in part order and runs the
  // SwiGLU epilogue.
  float *part_buf;
  int part_slots;
  int *part_cnt;
  int E, d, F;
  bf16 *act;   // [item][F/64] tiles: SwiGLU output rows
  bf16 *y;     // [rows][d]
  int *err;
};

constexpr int kTileElems = 128 * 64;

__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Named barrier 1 over the epilogue warps; epi_any also ORs a predicate over them.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;\n" ::"n"(kFfnEpiThreads) : "memory"); }
__device__ __forceinline__ bool epi_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kFfnEpiThreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(b)) : "memory");
}

// D (+)= A B^T with e4m3 A and B (kind::f8f6f4, K = 32 per instruction, the
// same 128-byte swizzled operand rows as the bf16 MMAs: 128 elements a row).
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum));
}

// Instruction descriptor: fp32 accumulator, e4m3 A and B (type code 0),
// both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ float swiglu_f(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *(uint32_t *)&v;
}

__global__ void __launch_bounds__(kFfnThreads, 1) moe_ffn_kernel(FfnArgs g) {
  using S = FfnSmem;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
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
  const int err_seen = threadIdx.x == 0 ? ld_err_word(g.err) : 0;
  if (threadIdx.x == 0) {
    *abort = 0;
    for (int s = 0; s < kFfnStages; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(acc_full + b, 1);
      tc::mbar_init(acc_empty + b, kFfnEpiWarps);  // one arrival per epilogue warp
    }
    for (int q = 0; q < kFfnQueue; ++q) {
      tc::mbar_init(q_full + q, 1);
      tc::mbar_init(q_empty + q, 1 + kFfnEpiWarps);  // the MMA thread and every epilogue warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  if (warp == kFfnMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     tc::smem_u32(tmem_slot)),
                 "r"(2u * kFfnPairCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  __syncwarp();  // lone-thread roles above: reconverge before the CTA-wide barrier
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the work list and the gathered rows come from earlier kernels
  pdl_trigger();
  if (threadIdx.x == 0 && err_seen) *abort = 1;

  const int n_items = *g.n_work;
  const int mA = (g.F + 127) / 128, mB = (g.d + 128 * kDownBlocks - 1) / (128 * kDownBlocks);
  const int nA = n_items * mA;
  // Gate/up units past a whole number of waves, when only a few (at most a
  // quarter of the grid), run split along K into S parts: the parts spread
  // over the SMs instead of a nearly empty extra wave of whole units.
  int n_ov = 0, S_ov = 1;
  // (only with at least one k-step per part)
  if (!g.fp8 && g.part_buf && nA > (int)gridDim.x && g.d / tc::kBK >= kFfnSplitParts) {
    const int rem = nA % (int)gridDim.x;
    if (rem > 0 && 4 * rem <= (int)gridDim.x && rem <= kFfnSplitUnits) {
      // the last part reads every part's sums: more parts, more bytes
      if (rem * kFfnSplitParts <= g.part_slots) {
        n_ov = rem;
        S_ov = kFfnSplitParts;
      }
    }
  }
  const int nA_full = nA - n_ov, nP = n_ov * S_ov;  // whole gate/up units first, then the parts
  const int n_units = nA_full + nP + n_items * mB;
  // gate/up k-steps: 64 bf16 or 128 e4m3 elements (128 bytes a row either way)
  const int KTA = g.fp8 ? g.d / 128 : g.d / tc::kBK, KTB = g.F / tc::kBK;
  auto a_tile = [&](int s, int j) { return base + (size_t)s * kFfnStageBytes + (size_t)j * kFfnATileBytes; };
  auto b_tile = [&](int s) { return base + (size_t)s * kFfnStageBytes + 2 * kFfnATileBytes; };

  if (warp == kFfnProducerWarp) {
    if (lane == 0) {
      int it = 0;
      for (int n = 0;; ++n) {
        const int q = n % kFfnQueue;
        if (n >= kFfnQueue) tc::mbar_wait(q_empty + q, ((n / kFfnQueue) - 1) & 1, g.err, 21, abort);
        // the first unit of every CTA is its block index (no atomic on the
        // way to the first copies); the counter hands out the rest
        const int u = *abort ? n_units : n == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(g.next, 1);
        UnitInfo inf;
        inf.u = u < n_units ? u : -1;
        if (inf.u >= 0) {
          inf.phase = u >= nA_full + nP;
          inf.part = -1;
          inf.ov = 0;
          inf.nparts = 1;
          int v, per = inf.phase ? mB : mA;
          if (inf.phase) {
            v = u - nA_full - nP;
          } else if (u < nA_full) {
            v = u;
          } else {  // part (u - nA_full) % S_ov of split unit (u - nA_full) / S_ov
            inf.ov = (u - nA_full) / S_ov;
            inf.part = (u - nA_full) - inf.ov * S_ov;
            inf.nparts = S_ov;
            v = nA_full + inf.ov;
          }
          inf.item = v / per;
          inf.mt = v - inf.item * per;
          const int KTu = inf.phase ? KTB : KTA;
          inf.kb = inf.part < 0 ? 0 : KTu * inf.part / S_ov;
          inf.ke = inf.part < 0 ? KTu : KTu * (inf.part + 1) / S_ov;
          const int e = g.work[2 * inf.item], n0 = g.work[2 * inf.item + 1];
          const int e0 = g.offs[e];
          inf.b_row = e0 + n0;
          inf.n_valid = min(kFfnBN, g.offs[e + 1] - e0 - n0);
          inf.e = e;
          inf.a_rows = inf.phase ? 128 : min(128, g.F - 128 * inf.mt);
          inf.n_acc = inf.phase ? min(kDownBlocks, g.d / 128 - kDownBlocks * inf.mt) : 2;
        }
        queue[q] = inf;
        mbar_arrive(q_full + q);  // release: the entry is visible to the waiting roles
        if (inf.u < 0) break;
        const int KT = inf.phase ? KTB : KTA;
        // weight tile kt of block j: a0 + j * a_blk + kt * a_kt
        const bf16 *a0;
        size_t a_blk;
        if (inf.phase) {
          a0 = g.wd + (size_t)inf.e * g.d * g.F + (size_t)(kDownBlocks * inf.mt) * 128 * g.F;
          a_blk = (size_t)128 * g.F;
        } else if (g.fp8) {  // e4m3 tiles: the bytes of bf16 tiles of half the columns
          const int dh = g.d / 2;
          a0 = (const bf16 *)g.wgu8 + (size_t)inf.e * 2 * g.F * dh + (size_t)128 * dh * inf.mt;
          a_blk = (size_t)g.F * dh;
        } else {
          a0 = g.wgu + (size_t)inf.e * 2 * g.F * g.d + (size_t)128 * g.d * inf.mt;
          a_blk = (size_t)g.F * g.d;
        }
        const size_t a_kt = (size_t)inf.a_rows * 64;
        const uint32_t a_bytes = (uint32_t)inf.a_rows * 128;
        const bf16 *bsrc = (inf.phase ? g.act : g.x) + (size_t)inf.item * KT * kTileElems;
        const uint32_t b_bytes = (uint32_t)((inf.n_valid + 7) & ~7) * 128;  // the item's valid rows
        const uint32_t tx = (uint32_t)inf.n_acc * a_bytes + b_bytes;
        auto load_a = [&](int s, int kt) {
          for (int j = 0; j < inf.n_acc; ++j)
            tc::bulk_load(a_tile(s, j), a0 + j * a_blk + kt * a_kt, a_bytes, full + s);
        };

        // Phase B: the first stages' weight tiles go out before the wait on act.
        const int pre = inf.phase ? min(KT, kFfnStages) : 0;
        for (int kt = 0; kt < pre; ++kt) {
          const int i = it + kt, s = i % kFfnStages, r = i / kFfnStages;
          if (r > 0) tc::mbar_wait(empty + s, (r - 1) & 1, g.err, 23, abort);
          if (*abort) break;
          tc::mbar_expect_tx(full + s, tx);
          load_a(s, kt);
        }
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
        int issued = it;  // stages whose copies went out (for the drain below)
        const int nk = inf.ke - inf.kb;  // the unit's k-steps (a split part: its K range)
        for (int kk = 0; kk < nk; ++kk) {
          const int kt = inf.kb + kk, i = it + kk, s = i % kFfnStages, r = i / kFfnStages;
          if (kk >= pre) {
            if (r > 0) tc::mbar_wait(empty + s, (r - 1) & 1, g.err, 23, abort);
            if (*abort) break;
            tc::mbar_expect_tx(full + s, tx);
            load_a(s, kt);
          } else if (*abort) {
            break;
          }
          tc::bulk_load(b_tile(s), bsrc + (size_t)kt * kTileElems, b_bytes, full + s);
          issued = i + 1;
        }
        if (*abort) {
          // Drain: wait (bounded) for the copies in flight, including weight
          // tiles requested ahead of the act wait, then hand over the end marker.
          const int last = max(issued, it + pre);
          for (int i = last - 1; i >= 0 && i >= last - kFfnStages; --i) {
            const long long t0 = clock64();
            while (!tc::mbar_try_wait(full + i % kFfnStages, (i / kFfnStages) & 1) &&
                   clock64() - t0 < tc::kWaitCycles) {
            }
          }
        }
        it += nk;
      }
    }
  } else if (warp == kFfnMmaWarp) {
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
        const uint32_t d0 = tmem + buf * kFfnPairCols, d1 = d0 + kFfnBN;
        const int n_mma = max(16, (inf.n_valid + 15) & ~15);
        const bool f8 = g.fp8 && inf.phase == 0;
        const uint32_t idesc = f8 ? idesc_e4m3(128, n_mma) : tc::idesc_bf16(128, n_mma);
        const int KT = inf.ke - inf.kb;  // the unit's k-steps (the first one starts the accumulators)
        for (int kt = 0; kt < KT; ++kt, ++it) {
          const int s = it % kFfnStages, r = it / kFfnStages;
          tc::mbar_wait(full + s, r & 1, g.err, 26, abort);
          tc::fence_after();
          const uint64_t adesc0 = tc::sw128_desc(tc::smem_u32(a_tile(s, 0)));
          const uint64_t adesc1 = tc::sw128_desc(tc::smem_u32(a_tile(s, 1)));
          const uint64_t bdesc = tc::sw128_desc(tc::smem_u32(b_tile(s)));
          if (f8) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {  // 32 e4m3 elements (32 bytes) per MMA
              mma_e4m3(d0, adesc0 + 2 * kk, bdesc + 2 * kk, idesc, (kt | kk) ? 1u : 0u);
              mma_e4m3(d1, adesc1 + 2 * kk, bdesc + 2 * kk, idesc, (kt | kk) ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < tc::kBK / 16; ++kk) {
              tc::mma_bf16(d0, adesc0 + 2 * kk, bdesc + 2 * kk, idesc, (kt | kk) ? 1u : 0u);
              if (inf.n_acc > 1) tc::mma_bf16(d1, adesc1 + 2 * kk, bdesc + 2 * kk, idesc, (kt | kk) ? 1u : 0u);
            }
          }
          tc::mma_commit(empty + s);
        }
        tc::mma_commit(acc_full + buf);
        mbar_arrive(q_empty + q);
      }
    }
  } else {
    // ---- epilogue: warps 0-7; lane = accumulator row, 64 token columns per warp
    __shared__ int split_last;  // written by thread 0, read by the epilogue after a barrier
    const int q4 = warp & 3, half = warp >> 2;
    const int lrow = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    for (int n = 0;; ++n) {
      const int q = n % kFfnQueue;
      tc::mbar_wait(q_full + q, (n / kFfnQueue) & 1, g.err, 27, abort);
      const UnitInfo inf = queue[q];
      // every epilogue warp takes the same decision (the named barriers below)
      if (epi_any(inf.u < 0 || *abort)) break;
      const int buf = n & 1;
      tc::mbar_wait(acc_full + buf, (n >> 1) & 1, g.err, 28, abort);
      tc::fence_after();
      const uint32_t tp = tmem + buf * kFfnPairCols + lane_off;
      // SwiGLU of feature f = 128 mt + lrow for the warp's token columns;
      // lanes 2i and 2i + 1 trade values so that each stores a bf16 pair
      // (features f, f + 1) of one token row into the act tile.
      const bool fok = lrow < inf.a_rows;
      const int fb = 128 * inf.mt + (lrow & ~1), cc = fb & 63;
      unsigned char *blk = inf.phase == 0
                               ? (unsigned char *)(g.act + ((size_t)inf.item * (g.F / 64) + (fb >> 6)) * kTileElems)
                               : nullptr;
      // gv, uv: the gate and up sums of NC consecutive token columns from col0
      auto store_act = [&](const auto &gv, const auto &uv, int col0) {
        constexpr int NC = sizeof(gv) / sizeof(uint32_t);
#pragma unroll
        for (int j = 0; j < NC / 2; ++j) {
          const float a0 = swiglu_f(__uint_as_float(gv[2 * j]), __uint_as_float(uv[2 * j]));
          const float a1 = swiglu_f(__uint_as_float(gv[2 * j + 1]), __uint_as_float(uv[2 * j + 1]));
          const float recv = __shfl_xor_sync(0xffffffffu, (lane & 1) ? a0 : a1, 1);
          const int t = col0 + 2 * j + (lane & 1);
          const uint32_t w = (lane & 1) ? pack_bf16x2(recv, a1) : pack_bf16x2(a0, recv);
          if (fok && t < inf.n_valid)
            *(uint32_t *)(blk + t * 128 + ((((cc >> 3) ^ (t & 7)) << 4) | ((cc & 7) << 1))) = w;
        }
      };
      // a split unit's part slots: [2 (gate, up)][32 groups of 4 token
      // columns][128 features][4] fp32 (a warp's 32 features of 4 columns:
      // 512 contiguous bytes, one 16-byte vector a lane)
      float *const pslot = inf.part >= 0 ? g.part_buf + (size_t)inf.ov * inf.nparts * (kFfnPartSlotBytes / 4) : nullptr;
      if (inf.phase == 0 && inf.part >= 0) {
        // one K range of a split gate/up unit: its sums into its slot
        float *pb = pslot + (size_t)inf.part * (kFfnPartSlotBytes / 4);
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          const int col0 = 64 * half + 32 * c;
          if (col0 >= inf.n_valid) break;
          uint32_t gv[32], uv[32];
          tc::tmem_ld32(tp + col0, gv);
          tc::tmem_ld32(tp + kFfnBN + col0, uv);
          tc::tmem_ld_wait(gv);
          tc::tmem_ld_wait(uv);
          float *const pg = pb + ((size_t)(col0 >> 2) * 128 + lrow) * 4;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            *(float4 *)(pg + 512 * j) = make_float4(__uint_as_float(gv[4 * j]), __uint_as_float(gv[4 * j + 1]),
                                                    __uint_as_float(gv[4 * j + 2]), __uint_as_float(gv[4 * j + 3]));
            *(float4 *)(pg + 128 * 128 + 512 * j) =
                make_float4(__uint_as_float(uv[4 * j]), __uint_as_float(uv[4 * j + 1]), __uint_as_float(uv[4 * j + 2]),
                            __uint_as_float(uv[4 * j + 3]));
          }
        }
      } else if (inf.phase == 0) {
        // fp8: this feature's gate and up exponents (the token rows' come per column)
        int kwg = 0, kwu = 0;
        if (g.fp8 && fok) {
          kwg = g.kw[((size_t)inf.e * 2) * g.F + 128 * inf.mt + lrow];
          kwu = g.kw[((size_t)inf.e * 2 + 1) * g.F + 128 * inf.mt + lrow];
        }
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          const int col0 = 64 * half + 32 * c;
          if (col0 >= inf.n_valid) break;
          uint32_t gv[32], uv[32];
          tc::tmem_ld32(tp + col0, gv);
          tc::tmem_ld32(tp + kFfnBN + col0, uv);
          const int kx_lane = g.fp8 && col0 + lane < inf.n_valid ? g.kx[inf.b_row + col0 + lane] : 0;
          tc::tmem_ld_wait(gv);
          tc::tmem_ld_wait(uv);
          if (g.fp8) {  // back to the rows' scales: exact powers of two
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int kx = __shfl_sync(0xffffffffu, kx_lane, j);
              gv[j] = __float_as_uint(ldexpf(__uint_as_float(gv[j]), kwg + kx));
              uv[j] = __float_as_uint(ldexpf(__uint_as_float(uv[j]), kwu + kx));
            }
          }
          store_act(gv, uv, col0);
        }
      } else {
        // y[row][256 mt + 128 a + lrow] (bf16) for the warp's token columns:
        // lanes 2i and 2i + 1 trade values so that each stores the feature
        // pair (f, f + 1) of one token row; per token column pair the warp
        // writes two 64-byte runs.
#pragma unroll 1
        for (int a = 0; a < inf.n_acc; ++a) {
          bf16 *dst = g.y + (size_t)inf.b_row * g.d + 128 * (kDownBlocks * inf.mt + a) + (lrow & ~1);
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            const int col0 = 64 * half + 32 * c;
            if (col0 >= inf.n_valid) break;
            uint32_t v[32];
            tc::tmem_ld32(tp + a * kFfnBN + col0, v);
            tc::tmem_ld_wait(v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float a0 = __uint_as_float(v[2 * j]), a1 = __uint_as_float(v[2 * j + 1]);
              const float recv = __shfl_xor_sync(0xffffffffu, (lane & 1) ? a0 : a1, 1);
              const int t = col0 + 2 * j + (lane & 1);
              const uint32_t w = (lane & 1) ? pack_bf16x2(recv, a1) : pack_bf16x2(a0, recv);
              if (t < inf.n_valid) *(uint32_t *)(dst + (size_t)t * g.d) = w;
            }
          }
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + buf);  // this warp's reads of the pair are done
      if (inf.phase == 0) {
        __threadfence();
        asm volatile("fence.proxy.async.global;\n" ::: "memory");
        epi_sync();
        bool publish = inf.part < 0;
        if (inf.part >= 0) {
          // the part's ticket; the last part (every other part's sums are
          // stored: their tickets came first) sums the parts in part order
          if (threadIdx.x == 0) split_last = atomicAdd(g.part_cnt + inf.ov, 1) == inf.nparts - 1;
          epi_sync();
          if (split_last) {
            __threadfence();
            // 16 token columns a pass: every part's gate and up vectors of
            // them in flight at once, then summed in part order
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              const int col0 = 64 * half + 16 * c;
              if (col0 >= inf.n_valid) break;
              float4 vg[kFfnSplitParts][4], vu[kFfnSplitParts][4];
#pragma unroll
              for (int q = 0; q < kFfnSplitParts; ++q) {
                const float *pb = pslot + (size_t)q * (kFfnPartSlotBytes / 4) + ((size_t)(col0 >> 2) * 128 + lrow) * 4;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  vg[q][k] = __ldcg((const float4 *)(pb + 512 * k));
                  vu[q][k] = __ldcg((const float4 *)(pb + 128 * 128 + 512 * k));
                }
              }
              uint32_t gv[16], uv[16];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                float4 sg = vg[0][k], su = vu[0][k];
#pragma unroll
                for (int q = 1; q < kFfnSplitParts; ++q) {
                  sg.x += vg[q][k].x, sg.y += vg[q][k].y, sg.z += vg[q][k].z, sg.w += vg[q][k].w;
                  su.x += vu[q][k].x, su.y += vu[q][k].y, su.z += vu[q][k].z, su.w += vu[q][k].w;
                }
                gv[4 * k] = __float_as_uint(sg.x), gv[4 * k + 1] = __float_as_uint(sg.y);
                gv[4 * k + 2] = __float_as_uint(sg.z), gv[4 * k + 3] = __float_as_uint(sg.w);
                uv[4 * k] = __float_as_uint(su.x), uv[4 * k + 1] = __float_as_uint(su.y);
                uv[4 * k + 2] = __float_as_uint(su.z), uv[4 * k + 3] = __float_as_uint(su.w);
              }
              store_act(gv, uv, col0);
            }
            __threadfence();
            asm volatile("fence.proxy.async.global;\n" ::: "memory");
            epi_sync();
            publish = true;
          }
        }
        if (publish && threadIdx.x == 0) atomicAdd(g.done + inf.item, 1);  // publish after every thread's stores
      }
      if (lane == 0) mbar_arrive(q_empty + q);  // this warp is done with the queue entry
    }
  }
  __syncwarp();  // lone-thread roles above: reconverge before the CTA-wide barrier
  tc::fence_before();
  __syncthreads();
  if (warp == kFfnMmaWarp) {
    tc::fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(2u * kFfnPairCols));
  }
}

// Rows of n_mat bf16 operand-tile matrices [R][C] (contiguous, R * C
// elements each) to e4m3 operand tiles (R * C bytes each) and their scale
// exponents [n_mat][R]: one warp per row, the row read twice (its maximum,
// then 16 elements per lane and step).
__global__ void quantize_rows_e4m3_kernel(const bf16 *src, uint8_t *dst, int *exps, int n_mat, int R, int C) {
  const int lane = threadIdx.x & 31;
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (gw >= (long long)n_mat * R) return;
  const int m = (int)(gw / R), r = (int)(gw - (long long)m * R);
  const bf16 *A = src + (size_t)m * R * C;
  uint8_t *B = dst + (size_t)m * R * C;
  float amax = 0.0f;
  for (int c = 8 * lane; c < C; c += 256) {
    const uint4 v = *(const uint4 *)(A + tiled_index(R, C, r, c));
    const __nv_bfloat162 *p2 = (const __nv_bfloat162 *)&v;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(p2[i]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const int k = e4m3_scale_exp(amax);
  for (int c = 16 * lane; c < C; c += 512) {
    uint4 v[2];
    v[0] = *(const uint4 *)(A + tiled_index(R, C, r, c));
    v[1] = *(const uint4 *)(A + tiled_index(R, C, r, c + 8));
    const __nv_bfloat162 *p2 = (const __nv_bfloat162 *)v;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = __bfloat1622float2(p2[2 * i]), b = __bfloat1622float2(p2[2 * i + 1]);
      w[i] = cvt_e4m3x2(ldexpf(a.x, -k), ldexpf(a.y, -k)) | (cvt_e4m3x2(ldexpf(b.x, -k), ldexpf(b.y, -k)) << 16);
    }
    *(uint4 *)(B + tiled_index_e4m3(R, C, r, c)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (lane == 0) exps[(size_t)m * R + r] = k;
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

cudaError_t quantize_rows_e4m3(const bf16 *src, uint8_t *dst, int *exps, int n_mat, int R, int C,
                               cudaStream_t st) {
  if (n_mat <= 0 || R <= 0) return cudaSuccess;
  if (C <= 0 || C % 128) return cudaErrorInvalidValue;
  const long long threads = (long long)n_mat * R * 32;
  quantize_rows_e4m3_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(src, dst, exps, n_mat, R, C);
  return cudaGetLastError();
}

size_t moe_ffn_part_slots() { return (size_t)ffn_num_sms(); }

cudaError_t moe_ffn(const bf16 *x_tiles, int rows, const bf16 *wgu, const bf16 *wd, const int *offs,
                    const int *work, const int *n_work, int max_work, int E, int d, int F, bf16 *act_tiles,
                    bf16 *y, int *err, cudaStream_t st, const Fp8Experts *fp8, float *part_buf,
                    int part_slots) {
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
  g.part_cnt = g.next + 1;  // kFfnSplitUnits tickets, zeroed by moe_scatter
  g.part_buf = part_buf;
  g.part_slots = part_buf ? part_slots : 0;
  g.E = E;
  g.d = d;
  g.F = F;
  g.act = act_tiles;
  g.y = y;
  g.err = err;
  if (fp8) {
    g.fp8 = 1;
    g.wgu8 = fp8->wgu8;
    g.kw = fp8->kw;
    g.kx = fp8->kx;
  }
  return launch_pdl(moe_ffn_kernel, dim3(ffn_num_sms()), dim3(kFfnThreads), FfnSmem::bytes, st, g);
}

}  // namespace dg
