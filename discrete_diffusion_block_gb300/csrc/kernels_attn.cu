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
#include <mutex>

#include "gemm_mma.cuh"
#include "internal.h"

namespace dg {

namespace {

constexpr int kRowsPerBlock = 64;  // 4 warps x 16 rows
constexpr int kKeysPerTile = 64;

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
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *(uint32_t *)&v;
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t *r, const void *p) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(s));
}

template <int HD>
__global__ void __launch_bounds__(128) attn_kernel(AttnParams p) {
  pdl_wait();
  pdl_trigger();
  constexpr int LDK = HD + 8;
  extern __shared__ __align__(16) unsigned char smem[];
  bf16 *Ks = (bf16 *)smem;                 // [2][64][LDK]
  bf16 *Vs = Ks + 2 * kKeysPerTile * LDK;  // [2][64][LDK]
  const int g = blockIdx.y, split = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rows_total = p.G * p.n_new;
  const int r_cta = blockIdx.x * kRowsPerBlock;
  const int n_keys = p.n_prefix + p.n_new;
  const int k_begin = split * p.keys_per_split;
  int k_end = min(n_keys, k_begin + p.keys_per_split);
  if (p.causal) {
    const int t_max = min(p.n_new - 1, (r_cta + kRowsPerBlock - 1) / p.G);
    k_end = min(k_end, p.n_prefix + t_max + 1);
  }
  const int rowA = r_cta + warp * 16 + (lane >> 2), rowB = rowA + 8;
  const bool okA = rowA < rows_total, okB = rowB < rows_total;
  const int limA = p.causal ? p.n_prefix + rowA / p.G : n_keys - 1;
  const int limB = p.causal ? p.n_prefix + rowB / p.G : n_keys - 1;

  auto qoff = [&](int row) { return ((size_t)(row / p.G) * p.Hq + g * p.G + row % p.G) * HD; };
  uint32_t qf[HD / 16][4];
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const int col = kk * 16 + 2 * (lane & 3);
    qf[kk][0] = okA ? *(const uint32_t *)(p.q + qoff(rowA) + col) : 0u;
    qf[kk][1] = okB ? *(const uint32_t *)(p.q + qoff(rowB) + col) : 0u;
    qf[kk][2] = okA ? *(const uint32_t *)(p.q + qoff(rowA) + col + 8) : 0u;
    qf[kk][3] = okB ? *(const uint32_t *)(p.q + qoff(rowB) + col + 8) : 0u;
  }

  auto load_tile = [&](int stage, int kb) {
    bf16 *ks = Ks + stage * kKeysPerTile * LDK;
    bf16 *vs = Vs + stage * kKeysPerTile * LDK;
    for (int c = tid; c < kKeysPerTile * (HD / 8); c += 128) {
      const int key = c / (HD / 8), ch = c % (HD / 8);
      const int j = kb * kKeysPerTile + key;
      const bool ok = j < k_end;
      size_t off = 0;
      if (ok) off = (((size_t)p.page_table[j / p.pg] * p.Hkv + g) * p.pg + j % p.pg) * HD + ch * 8;
      cp_async16(ks + key * LDK + ch * 8, p.k_pool + off, ok);
      cp_async16(vs + key * LDK + ch * 8, p.v_pool + off, ok);
    }
  };

  float o[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i)
#pragma unroll
    for (int r = 0; r < 4; ++r) o[i][r] = 0.0f;
  const float NEG = __int_as_float(0xff800000);
  float mA = NEG, mB = NEG, lA = 0.0f, lB = 0.0f;

  const int kb0 = k_begin / kKeysPerTile;
  const int kb1 = k_end > k_begin ? ceil_div(k_end, kKeysPerTile) : kb0;
  if (kb0 < kb1) load_tile(0, kb0);
  cp_async_commit();
  for (int kb = kb0; kb < kb1; ++kb) {
    const int stage = (kb - kb0) & 1;
    if (kb + 1 < kb1) load_tile(stage ^ 1, kb + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const bf16 *ks = Ks + stage * kKeysPerTile * LDK;
    const bf16 *vs = Vs + stage * kKeysPerTile * LDK;
    float s[8][4];
#pragma unroll
    for (int jn = 0; jn < 8; ++jn)
#pragma unroll
      for (int r = 0; r < 4; ++r) s[jn][r] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk)
#pragma unroll
      for (int jn = 0; jn < 8; ++jn) {
        const bf16 *kp = ks + (jn * 8 + (lane >> 2)) * LDK + kk * 16 + 2 * (lane & 3);
        uint32_t b[2] = {*(const uint32_t *)kp, *(const uint32_t *)(kp + 8)};
        mma_bf16_16816(s[jn], qf[kk], b);
      }
    float mxA = NEG, mxB = NEG;
#pragma unroll
    for (int jn = 0; jn < 8; ++jn)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int j = kb * kKeysPerTile + jn * 8 + 2 * (lane & 3) + (r & 1);
        const bool vis = j < k_end && j <= (r < 2 ? limA : limB);
        const float v = vis ? s[jn][r] * p.scale_log2 : NEG;
        s[jn][r] = v;
        if (r < 2) mxA = fmaxf(mxA, v); else mxB = fmaxf(mxB, v);
      }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, off));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, off));
    }
    const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
    const float uA = nA == NEG ? 0.0f : nA, uB = nB == NEG ? 0.0f : nB;
    const float aA = exp2f(mA - uA), aB = exp2f(mB - uB);
    mA = nA;
    mB = nB;
    lA *= aA;
    lB *= aB;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      o[i][0] *= aA; o[i][1] *= aA;
      o[i][2] *= aB; o[i][3] *= aB;
    }
    uint32_t pf[4][4];
#pragma unroll
    for (int jn = 0; jn < 8; ++jn) {
      const float p0 = exp2f(s[jn][0] - uA), p1 = exp2f(s[jn][1] - uA);
      const float p2 = exp2f(s[jn][2] - uB), p3 = exp2f(s[jn][3] - uB);
      lA += p0 + p1;
      lB += p2 + p3;
      pf[jn >> 1][(jn & 1) * 2 + 0] = pack_bf16(p0, p1);
      pf[jn >> 1][(jn & 1) * 2 + 1] = pack_bf16(p2, p3);
    }
#pragma unroll
    for (int ks2 = 0; ks2 < 4; ++ks2)
#pragma unroll
      for (int dp = 0; dp < HD / 16; ++dp) {
        const int key = ks2 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int dim = dp * 16 + (lane >> 4) * 8;
        uint32_t r[4];
        ldsm_x4_trans(r, vs + key * LDK + dim);
        uint32_t b0[2] = {r[0], r[1]}, b1[2] = {r[2], r[3]};
        mma_bf16_16816(o[2 * dp], pf[ks2], b0);
        mma_bf16_16816(o[2 * dp + 1], pf[ks2], b1);
      }
    __syncthreads();
  }
  cp_async_wait<0>();
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    lA += __shfl_xor_sync(0xffffffffu, lA, off);
    lB += __shfl_xor_sync(0xffffffffu, lB, off);
  }
  if (p.out) {
    const float iA = lA > 0.0f ? 1.0f / lA : 0.0f, iB = lB > 0.0f ? 1.0f / lB : 0.0f;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      const int col = i * 8 + 2 * (lane & 3);
      if (okA) *(uint32_t *)(p.out + qoff(rowA) + col) = pack_bf16(o[i][0] * iA, o[i][1] * iA);
      if (okB) *(uint32_t *)(p.out + qoff(rowB) + col) = pack_bf16(o[i][2] * iB, o[i][3] * iB);
    }
  } else {
    const size_t base = ((size_t)split * p.Hkv + g) * rows_total;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      const int col = i * 8 + 2 * (lane & 3);
      if (okA) {
        float *d = p.o_part + (base + rowA) * HD + col;
        d[0] = o[i][0];
        d[1] = o[i][1];
      }
      if (okB) {
        float *d = p.o_part + (base + rowB) * HD + col;
        d[0] = o[i][2];
        d[1] = o[i][3];
      }
    }
    if ((lane & 3) == 0) {
      if (okA) { p.ml_part[(base + rowA) * 2] = mA; p.ml_part[(base + rowA) * 2 + 1] = lA; }
      if (okB) { p.ml_part[(base + rowB) * 2] = mB; p.ml_part[(base + rowB) * 2 + 1] = lB; }
    }
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
  int splits = ceil_div(2 * 152, base);
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

cudaError_t attention(const bf16 *q, const bf16 *k_pool, const bf16 *v_pool, const int *page_table,
                      const AttnShape &s, bf16 *out, void *ws, size_t ws_bytes, cudaStream_t st) {
  if (s.n_new <= 0) return cudaSuccess;
  if ((s.hd != 64 && s.hd != 128) || s.Hq % s.Hkv != 0 || s.pg % kKeysPerTile != 0)
    return cudaErrorInvalidValue;
  const SplitPlan pl = plan_splits(s);
  AttnParams p;
  p.q = q;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.page_table = page_table;
  p.n_prefix = s.n_prefix;
  p.n_new = s.n_new;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.G = s.Hq / s.Hkv;
  p.pg = s.pg;
  p.causal = s.causal;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)s.hd));
  p.keys_per_split = pl.keys_per_split;
  const int rows_total = p.G * s.n_new;
  if (pl.splits > 1) {
    if (ws_bytes < attention_workspace_bytes(s) || ws == nullptr) return cudaErrorInvalidValue;
    p.out = nullptr;
    p.o_part = (float *)ws;
    p.ml_part = p.o_part + (size_t)pl.splits * s.Hkv * rows_total * s.hd;
  } else {
    p.out = out;
    p.o_part = p.ml_part = nullptr;
  }
  dim3 grid(ceil_div(rows_total, kRowsPerBlock), s.Hkv, pl.splits);
  const size_t smem = (size_t)4 * kKeysPerTile * (s.hd + 8) * sizeof(bf16);
  static unsigned long long attr_set[2] = {0, 0};  // per device, per head size
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int which = s.hd == 128 ? 1 : 0;
  if (dev >= 64 || !((attr_set[which] >> dev) & 1ull)) {
    e = which ? cudaFuncSetAttribute(attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
              : cudaFuncSetAttribute(attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set[which] |= 1ull << dev;
  }
  e = which ? launch_pdl(attn_kernel<128>, grid, dim3(128), smem, st, p)
            : launch_pdl(attn_kernel<64>, grid, dim3(128), smem, st, p);
  if (e != cudaSuccess) return e;
  if (pl.splits > 1)
    e = launch_pdl(attn_combine_kernel, dim3(rows_total, s.Hkv), dim3(128), 0, st, (const float *)p.o_part,
                   (const float *)p.ml_part, pl.splits, s.Hkv, rows_total, p.G, s.Hq, s.hd, out);
  return e;
}

}  // namespace dg
