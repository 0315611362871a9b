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
// The kernel is a tcgen05 tensor-core kernel with two passes over the
// block's key range:
//   pass 1  S = Q K^T per 128-key tile (TMEM), running row max m;
//   pass 2  S again, P = 2^(S*scale - m) as bf16 into shared memory, row sum
//           l in fp32, O += P V (TMEM) -- with m final, O is never rescaled.
// The second QK^T costs a third more tensor work and saves the read-modify-
// write of the accumulator that a one-pass online softmax needs.  Roles:
// warp 0 streams Q once and the K (and V) tiles of each pass through a
// two-slot ring with TMA (Q through a 4-D map that packs the G heads of a
// token as consecutive rows; K and V as 64-key boxes of their pages); warp 1
// issues the MMAs (V is the N-contiguous "MN-major" B operand of P V); warps
// 2-5 hold one row each and do the softmax on the accumulator rows they read
// from TMEM.
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
  bf16 *out;
  float *o_part;   // [splits][Hkv][rows][HD] (split launches)
  float *ml_part;  // [splits][Hkv][rows][2]
  int *err;        // device error word (bounded waits, bad page indices), may be null
  int n_pages;     // physical pages of the pools, 0 when unknown
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *(uint32_t *)&v;
}


constexpr int kAttnThreads = 192;
constexpr int kAttnSlotHalfBytes = 64 * 128;  // 64 keys x 64 hd bf16 (one TMA box)

template <int HD>
struct AttnSmem {
  static constexpr int HB = HD / 64;                       // 64-wide hd blocks
  static constexpr size_t q = 0;                           // HB x [128 rows][64] bf16
  static constexpr size_t q_bytes = (size_t)HB * 16384;
  static constexpr size_t k_bytes = (size_t)HB * 16384;    // HB x [128 keys][64]
  static constexpr size_t v_bytes = (size_t)HB * 16384;    // HB x [128 keys][64] (N-contiguous B)
  static constexpr size_t slot_bytes = k_bytes + v_bytes;
  static constexpr size_t ring = q + q_bytes;              // 2 slots
  static constexpr size_t pbuf = ring + 2 * slot_bytes;    // 2 x [128 rows][64 keys] bf16
  static constexpr size_t pages = pbuf + 32768;            // page of every 64-key half (ints)
  static constexpr int kMaxHalves = 1024;
  static constexpr size_t bars = pages + kMaxHalves * 4;
  // q_full, kv_full[2], kv_empty[2], s_full[2], s_empty[2], p_full, p_empty, o_full; TMEM slot; abort
  static constexpr size_t bytes = bars + 12 * 8 + 16 + 1024;
};

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

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, AttnParams p) {
  using S = AttnSmem<HD>;
  constexpr int HB = S::HB;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  int *pages = (int *)(base + S::pages);
  uint64_t *q_full = (uint64_t *)(base + S::bars);
  uint64_t *kv_full = q_full + 1, *kv_empty = kv_full + 2;
  uint64_t *s_full = kv_empty + 2, *s_empty = s_full + 2;
  uint64_t *p_full = s_empty + 2, *p_empty = p_full + 1, *o_full = p_empty + 1;
  uint32_t *tmem_slot = (uint32_t *)(o_full + 1);
  volatile int *abort = (volatile int *)(tmem_slot + 1);
  auto k_tile = [&](int slot) { return base + S::ring + (size_t)slot * S::slot_bytes; };
  auto v_tile = [&](int slot) { return base + S::ring + (size_t)slot * S::slot_bytes + S::k_bytes; };

  const int g = blockIdx.y, split = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_total = p.G * p.n_new;
  const int r_cta = blockIdx.x * 128;
  const int n_keys = p.n_prefix + p.n_new;
  const int k_begin = split * p.keys_per_split;
  int k_end = min(n_keys, k_begin + p.keys_per_split);
  if (p.causal) {
    const int t_max = min(p.n_new - 1, (r_cta + 127) / p.G);
    k_end = min(k_end, p.n_prefix + t_max + 1);
  }
  const int n_kt = k_end > k_begin ? ceil_div(k_end - k_begin, 128) : 0;

  if (threadIdx.x == 0) {
    *abort = 0;
    tc::mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(kv_full + i, 1);
      tc::mbar_init(kv_empty + i, 1);
      tc::mbar_init(s_full + i, 1);
      tc::mbar_init(s_empty + i, 4);
    }
    tc::mbar_init(p_full, 4);
    tc::mbar_init(p_empty, 1);
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
  pdl_wait();
  pdl_trigger();
  // physical page of every 64-key half of this block's range
  const int n_halves = 2 * n_kt;
  for (int i = threadIdx.x; i < n_halves && i < S::kMaxHalves; i += blockDim.x) {
    const int key0 = k_begin + 64 * i;
    int pg_i = key0 < k_end ? p.page_table[key0 / p.pg] : -1;
    if (pg_i >= 0 && p.n_pages > 0 && pg_i >= p.n_pages) {  // a page index outside the pool: skip it
      if (p.err) atomicExch(p.err, 39);
      pg_i = -1;
    }
    pages[i] = pg_i;
  }
  if (threadIdx.x == 0 && p.err && *(volatile int *)p.err) *abort = 1;
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_s = tmem, t_o = tmem + 256;  // S double buffer: columns [0,128) [128,256); O: [256, 256+HD)

  if (warp == 0) {
    if (lane == 0 && n_kt > 0) {
      tc::mbar_expect_tx(q_full, (uint32_t)S::q_bytes);
      for (int b = 0; b < HB; ++b) {
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes "
            "[%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(tc::smem_u32(base + S::q + (size_t)b * 16384)),
            "l"((uint64_t)&tq), "r"(64 * b), "r"(0), "r"(g), "r"(r_cta / p.G), "r"(tc::smem_u32(q_full))
            : "memory");
      }
      // two passes over the tiles; pass 1 loads K only
      int issued = 0;
      for (int i = 0; i < 2 * n_kt; ++i, issued = i) {
        const int pass = i >= n_kt, kt = pass ? i - n_kt : i, slot = i & 1;
        if (i >= 2) tc::mbar_wait(kv_empty + slot, ((i >> 1) - 1) & 1, p.err, 31, abort);
        if (*abort) break;
        tc::mbar_expect_tx(kv_full + slot, (pass ? 4u : 2u) * HB * kAttnSlotHalfBytes);
        for (int h = 0; h < 2; ++h) {
          // a half past the block's last key is fetched from rows before the
          // tensor's start: the fill value (zero) lands in its slot
          const int pg_i = pages[2 * kt + h];
          const int key0 = k_begin + 128 * kt + 64 * h;
          const int row = pg_i < 0 ? -64 : (pg_i * p.Hkv + g) * p.pg + key0 % p.pg;
          for (int b = 0; b < HB; ++b) {
            tc::tma_load_2d(k_tile(slot) + (size_t)b * 16384 + h * kAttnSlotHalfBytes, &tk, 64 * b, row, kv_full + slot);
            if (pass)
              tc::tma_load_2d(v_tile(slot) + (size_t)b * 16384 + h * kAttnSlotHalfBytes, &tv, 64 * b, row, kv_full + slot);
          }
        }
      }
      if (*abort) {  // drain the copies still in flight: the last load of each slot (bounded)
        for (int i = issued - 1; i >= 0 && i >= issued - 2; --i) {
          const long long t0 = clock64();
          while (!tc::mbar_try_wait(kv_full + (i & 1), (i >> 1) & 1) && clock64() - t0 < tc::kWaitCycles) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && n_kt > 0) {
      const uint32_t idesc_s = tc::idesc_bf16(128, 128);
      const uint32_t idesc_o = tc::idesc_bf16(128, HD) | (1u << 16);  // B (V) N-contiguous
      tc::mbar_wait(q_full, 0, p.err, 32, abort);
      auto issue_s = [&](int i) {  // S[i & 1] = Q K^T of ring load i
        const int slot = i & 1, buf = i & 1;
        if (i >= 2) tc::mbar_wait(s_empty + buf, ((i >> 1) - 1) & 1, p.err, 33, abort);
        tc::mbar_wait(kv_full + slot, (i >> 1) & 1, p.err, 34, abort);
        tc::fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint64_t adesc = tc::sw128_desc(tc::smem_u32(base + S::q + (size_t)(kk >> 2) * 16384)) + 2 * (kk & 3);
          const uint64_t bdesc = tc::sw128_desc(tc::smem_u32(k_tile(slot) + (size_t)(kk >> 2) * 16384)) + 2 * (kk & 3);
          tc::mma_bf16(t_s + buf * 128, adesc, bdesc, idesc_s, kk ? 1u : 0u);
        }
        tc::mma_commit(s_full + buf);
      };
      for (int i = 0; i < n_kt; ++i) {  // pass 1
        issue_s(i);
        tc::mma_commit(kv_empty + (i & 1));
      }
      issue_s(n_kt);
      for (int kt = 0; kt < n_kt; ++kt) {  // pass 2
        const int i = n_kt + kt, slot = i & 1;
        if (kt + 1 < n_kt) issue_s(i + 1);
        tc::mbar_wait(p_full, kt & 1, p.err, 35, abort);
        tc::fence_after();
        const unsigned char *pb = base + S::pbuf;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // 128 keys, 16 per MMA
          const uint64_t adesc = tc::sw128_desc(tc::smem_u32(pb + (size_t)(kk >> 2) * 16384)) + 2 * (kk & 3);
          const uint64_t bdesc = mn_desc(tc::smem_u32(v_tile(slot))) + (uint64_t)kk * (2048 >> 4);
          tc::mma_bf16(t_o, adesc, bdesc, idesc_o, (kt | kk) ? 1u : 0u);
        }
        tc::mma_commit(p_empty);
        tc::mma_commit(kv_empty + slot);
      }
      tc::mma_commit(o_full);
    }
  } else {
    // ---- softmax warps: thread = query row ----------------------------------
    const int q4 = warp & 3, row = 32 * q4 + lane, r = r_cta + row;
    const bool ok = r < rows_total;
    const int lim = p.causal ? p.n_prefix + (ok ? r / p.G : 0) : n_keys - 1;
    const float NEG = __int_as_float(0xff800000);
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    float m = NEG, l = 0.0f;
    for (int i = 0; i < 2 * n_kt; ++i) {
      const int pass = i >= n_kt, kt = pass ? i - n_kt : i, buf = i & 1;
      tc::mbar_wait(s_full + buf, (i >> 1) & 1, p.err, 36, abort);
      tc::fence_after();
      const int key_base = k_begin + 128 * kt;
      uint32_t x[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld32(t_s + buf * 128 + lane_off + 32 * c, x[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld_wait(x[c]);  // ties every loaded register to the wait
      tc::fence_before();
      __syncwarp();
      if (lane == 0) attn_arrive(s_empty + buf);
      if (!pass) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int key = key_base + 32 * c + j;
            if (key < k_end && key <= lim) m = fmaxf(m, __uint_as_float(x[c][j]) * p.scale_log2);
          }
      } else {
        const float mu = m == NEG ? 0.0f : m;
        uint32_t pk[4][16];
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const int key = key_base + 32 * c + j;
            const float p0 = (key < k_end && key <= lim) ? exp2f(__uint_as_float(x[c][j]) * p.scale_log2 - mu) : 0.0f;
            const float p1 = (key + 1 < k_end && key + 1 <= lim) ? exp2f(__uint_as_float(x[c][j + 1]) * p.scale_log2 - mu) : 0.0f;
            l += p0 + p1;
            pk[c][j >> 1] = pack_bf16(p0, p1);
          }
        // previous P V done with the buffer?
        if (kt > 0) tc::mbar_wait(p_empty, (kt - 1) & 1, p.err, 37, abort);
        unsigned char *prow = base + S::pbuf + (size_t)row * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int h = c >> 1;  // keys 0-63 in box 0, 64-127 in box 1
#pragma unroll
          for (int u = 0; u < 4; ++u) {  // 16-byte chunks of this 32-key group
            const int chunk = (c & 1) * 4 + u;
            uint4 v = make_uint4(pk[c][4 * u], pk[c][4 * u + 1], pk[c][4 * u + 2], pk[c][4 * u + 3]);
            *(uint4 *)(prow + (size_t)h * 16384 + ((chunk ^ (row & 7)) << 4)) = v;
          }
        }
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        __syncwarp();
        if (lane == 0) attn_arrive(p_full);
      }
    }
    // ---- output -------------------------------------------------------------
    if (n_kt > 0) {
      tc::mbar_wait(o_full, 0, p.err, 38, abort);
      tc::fence_after();
    }
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    const size_t qrow = ok ? (((size_t)(r / p.G) * p.Hq + g * p.G + r % p.G) * HD) : 0;
    const size_t prow_o = ((size_t)split * p.Hkv + g) * rows_total + r;
#pragma unroll 1
    for (int c = 0; c < HD / 32; ++c) {
      uint32_t v[32];
      if (n_kt > 0) {
        tc::tmem_ld32(t_o + lane_off + 32 * c, v);
        tc::tmem_ld_wait(v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0u;
      }
      if (!ok) continue;
      if (p.out) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          uint4 w;
          w.x = pack_bf16(__uint_as_float(v[j]) * inv, __uint_as_float(v[j + 1]) * inv);
          w.y = pack_bf16(__uint_as_float(v[j + 2]) * inv, __uint_as_float(v[j + 3]) * inv);
          w.z = pack_bf16(__uint_as_float(v[j + 4]) * inv, __uint_as_float(v[j + 5]) * inv);
          w.w = pack_bf16(__uint_as_float(v[j + 6]) * inv, __uint_as_float(v[j + 7]) * inv);
          *(uint4 *)(p.out + qrow + 32 * c + j) = w;
        }
      } else {
        float4 *d = (float4 *)(p.o_part + prow_o * HD + 32 * c);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          d[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]), __uint_as_float(v[4 * j + 2]),
                             __uint_as_float(v[4 * j + 3]));
      }
    }
    if (ok && !p.out) {
      p.ml_part[prow_o * 2] = m;
      p.ml_part[prow_o * 2 + 1] = l;
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(512u));
  }
}

// Merge the split-KV partial states of one (row, KV head): weights 2^(m_s - m*).
__global__ void attn_combine_kernel(const float *o_part, const float *ml_part, int splits, int Hkv,
                                    int rows_total, int G, int Hq, int HD, bf16 *out) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x, g = blockIdx.y;
  const float NEG = __int_as_float(0xff800000);
  float mx = NEG;
  for (int s = 0; s < splits; ++s) mx = fmaxf(mx, ml_part[(((size_t)s * Hkv + g) * rows_total + row) * 2]);
  float L = 0.0f;
  for (int s = 0; s < splits; ++s) {
    const size_t b = ((size_t)s * Hkv + g) * rows_total + row;
    const float m = ml_part[b * 2];
    if (m != NEG) L += exp2f(m - mx) * ml_part[b * 2 + 1];
  }
  const int t = row / G, h = g * G + row % G;
  for (int c = threadIdx.x; c < HD; c += blockDim.x) {
    float acc = 0.0f;
    for (int s = 0; s < splits; ++s) {
      const size_t b = ((size_t)s * Hkv + g) * rows_total + row;
      const float m = ml_part[b * 2];
      if (m != NEG) acc += exp2f(m - mx) * o_part[b * HD + c];
    }
    out[((size_t)t * Hq + h) * HD + c] = __float2bfloat16_rn(acc / L);
  }
}

struct SplitPlan {
  int splits, keys_per_split;
};

SplitPlan plan_splits(const AttnShape &s) {
  const int G = s.Hq / s.Hkv;
  const int base = s.Hkv * ceil_div(G * s.n_new, kRowsPerBlock);
  const int n_keys = s.n_prefix + s.n_new;
  const int n_kb = ceil_div(n_keys, kKeysPerTile);
  int splits = 148 / base;  // about one wave: one 192 KB block per SM
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

// Fixed split-KV scratch for the entry point that must not allocate.  It is
// a file-scope device array, so every GPU that loads the library holds it
// for the life of the process.  Host code may not pass the symbol itself to
// a kernel (on the host it only names a stand-in); its device address is
// looked up once per device, with that device current.
static __device__ __align__(256) unsigned char g_attention_scratch[kAttentionFixedScratchBytes];

cudaError_t attention_fixed_scratch(void **ptr) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void *addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attention_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

int attention_launch_count(const AttnShape &s) {
  if (s.n_new <= 0) return 0;
  return plan_splits(s).splits > 1 ? 2 : 1;
}

size_t attention_workspace_bytes(const AttnShape &s) {
  if (s.n_new <= 0 || s.Hkv < 1) return 0;
  const SplitPlan pl = plan_splits(s);
  if (pl.splits <= 1) return 0;
  const size_t rows = (size_t)(s.Hq / s.Hkv) * s.n_new;
  return (size_t)pl.splits * s.Hkv * rows * (s.hd + 2) * sizeof(float);
}

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
cudaError_t launch_attn(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const AttnParams &p, dim3 grid, cudaStream_t st) {
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
  return launch_pdl(attn_tc_kernel<HD>, grid, dim3(kAttnThreads), S::bytes, st, tq, tk, tv, p);
}

}  // namespace

cudaError_t attention(const bf16 *q, const bf16 *k_pool, const bf16 *v_pool, const int *page_table,
                      const AttnShape &s, bf16 *out, void *ws, size_t ws_bytes, cudaStream_t st,
                      int *err) {
  if (s.n_new <= 0) return cudaSuccess;
  if ((s.hd != 64 && s.hd != 128) || s.Hq % s.Hkv != 0 || s.pg % 64 != 0) return cudaErrorInvalidValue;
  const int G = s.Hq / s.Hkv;
  if (128 % G) return cudaErrorInvalidValue;
  const SplitPlan pl = plan_splits(s);
  if (pl.keys_per_split > 64 * AttnSmem<128>::kMaxHalves) return cudaErrorInvalidValue;
  AttnParams p;
  p.q = q;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.page_table = page_table;
  p.n_prefix = s.n_prefix;
  p.n_new = s.n_new;
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
  if (pl.splits > 1) {
    if (ws_bytes < attention_workspace_bytes(s) || ws == nullptr) return cudaErrorInvalidValue;
    p.out = nullptr;
    p.o_part = (float *)ws;
    p.ml_part = p.o_part + (size_t)pl.splits * s.Hkv * rows_total * s.hd;
  } else {
    p.out = out;
    p.o_part = p.ml_part = nullptr;
  }
  // Q [T][Hq][hd] as a 4-D tensor (hd, G, Hkv, T): a box of 64 x G x 1 x 128/G
  // lands as 128 rows (token, head of the group) of 128 bytes.
  CUtensorMap tq, tk, tv;
  {
    const uint64_t dims[4] = {(uint64_t)s.hd, (uint64_t)G, (uint64_t)s.Hkv, (uint64_t)s.n_new};
    const uint64_t strides[3] = {(uint64_t)s.hd * 2, (uint64_t)G * s.hd * 2, (uint64_t)s.Hq * s.hd * 2};
    const uint32_t box[4] = {64, (uint32_t)G, 1, (uint32_t)(128 / G)};
    cudaError_t e = attn_map(&tq, q, 4, dims, strides, box);
    if (e != cudaSuccess) return e;
  }
  // K and V pools [pages][Hkv][pg][hd] as [pages * Hkv * pg][hd], 64-key boxes.
  // The pool size is not part of the call, so the map's row extent is set far
  // beyond any pool; only rows of pages the page table names are requested.
  {
    const uint64_t rows = s.n_pages > 0 ? (uint64_t)s.n_pages * s.Hkv * s.pg : (uint64_t)1 << 28;
    const uint64_t dims[2] = {(uint64_t)s.hd, rows};
    const uint64_t strides[1] = {(uint64_t)s.hd * 2};
    const uint32_t box[2] = {64, 64};
    cudaError_t e = attn_map(&tk, k_pool, 2, dims, strides, box);
    if (e != cudaSuccess) return e;
    e = attn_map(&tv, v_pool, 2, dims, strides, box);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(ceil_div(rows_total, kRowsPerBlock), s.Hkv, pl.splits);
  cudaError_t e = s.hd == 128 ? launch_attn<128>(tq, tk, tv, p, grid, st) : launch_attn<64>(tq, tk, tv, p, grid, st);
  if (e != cudaSuccess) return e;
  if (pl.splits > 1)
    e = launch_pdl(attn_combine_kernel, dim3(rows_total, s.Hkv), dim3(128), 0, st, (const float *)p.o_part,
                   (const float *)p.ml_part, pl.splits, s.Hkv, rows_total, p.G, s.Hq, s.hd, out);
  return e;
}

}  // namespace dg
