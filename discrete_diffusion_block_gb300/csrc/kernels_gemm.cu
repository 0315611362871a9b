// Projection, expert and LM-head GEMMs of the decoder (tcgen05, gemm_tc.cuh)
// with their fused epilogues.  Weights are the A operand (rows = output
// features, 128 per MMA) for every projection -- the token count is the short
// side -- except the LM head, whose epilogue needs a token's whole 256-wide
// vocab tile in one row.
#include <cudaTypedefs.h>

#include <mutex>
#include <unordered_map>

#include "gemm_tc.cuh"
#include "internal.h"

namespace dg {

namespace {

// q/k/v projection: RoPE (rotate-half pairs (j, j+hd/2)) on q and k at each
// row's absolute position (its request's first position + the row's index
// within the request); q to [T][Hq*hd]; k and v straight into the paged pool
// slice of this layer, through the row's request's page-table slice.  The tile holds whole heads (128 rows are
// one head of 128 or two of 64).  Tokens are taken 64 at a time: their
// cos/sin rows and page slots are staged in shared memory, then each thread
// rotates two adjacent pairs (j, j+1) and (j+hd/2, j+1+hd/2) of one token and
// stores them as bf16x2.
struct EpiQkv {
  static constexpr int kTok = 64, kMaxHalf = 64;
  static constexpr size_t extra_smem =
      (size_t)kTok * kMaxHalf * 2 * sizeof(float) + kTok * sizeof(long long) + kTok * sizeof(int);
  QkvOut o;
  // Stage the cos/sin rows and page slots of tokens t0 .. t0 + nt - 1 of the
  // tile with threads tid of nthr (64 or 128; nt <= kTok <= nthr), all loads
  // in flight at once.
  __device__ void stage(const TileCtx &c, unsigned char *extra, int t0, int nt, int tid, int nthr) const {
    const int half = o.hd >> 1, q4 = half >> 2, n4 = nt * q4;
    float *cs = (float *)extra;
    float *sn = cs + kTok * kMaxHalf;
    long long *slot = (long long *)(sn + kTok * kMaxHalf);
    const int rw = c.n0 + t0 + tid, ps = o.rows.pos(rw);
    const long long page =
        tid < nt ? (long long)o.page_table[o.rows.req(rw) * o.rows.pages_per_req + ps / o.pg] : 0;
    for (int i0 = 0; i0 < n4; i0 += 8 * nthr) {
      float4 rc[8], rs[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + tid + nthr * u;
        if (i < n4) {
          const int t = i / q4, j4 = i - t * q4;
          const size_t p = (size_t)o.rows.pos(c.n0 + t0 + t);
          rc[u] = ((const float4 *)(o.cos_t + p * half))[j4];
          rs[u] = ((const float4 *)(o.sin_t + p * half))[j4];
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + tid + nthr * u;
        if (i < n4) {
          const int t = i / q4, j4 = i - t * q4;
          ((float4 *)(cs + t * half))[j4] = rc[u];
          ((float4 *)(sn + t * half))[j4] = rs[u];
        }
      }
    }
    if (tid < nt) {
      slot[tid] = page * o.Hkv * o.pg * o.hd + (long long)(ps % o.pg) * 64;
      ((int *)(slot + kTok))[tid] = ps & 7;  // the pool row's chunk swizzle
    }
  }
  // Split-K with slices of up to kTok tokens: the slice's cos/sin rows and
  // page slots are staged by prepare() into memory of their own, before the
  // wait on the previous kernel (tables and page table are inputs of the
  // step, not outputs of earlier kernels).
  static constexpr bool kPrepEarly = true;
  static constexpr bool kDirect = false;  // RoPE pairs rows f and f + hd/2: through the shared tile
  static constexpr size_t prep_bytes(int w) { return w <= kTok ? extra_smem : 0; }
  __device__ void direct(const TileCtx &, int, int, const float (&)[32], unsigned char *) const {}
  __device__ void prepare(const TileCtx &c, unsigned char *extra, int tid, int nthr) const {
    stage(c, extra, 0, min(kTok, c.n_valid), tid, nthr);
  }
  __device__ void operator()(float *tile, int ldc, const TileCtx &c, unsigned char *extra) const {
    const int hd = o.hd, half = hd >> 1, qdim = o.Hq * hd, kdim = o.Hkv * hd;
    const int pairs_log = hd == 128 ? 5 : 4;  // half/2 = 32 or 16 pairs of pairs per head
    const int units = (c.m_valid / hd) << pairs_log;
    float *cs = (float *)extra;                           // [kTok][half]
    float *sn = cs + kTok * kMaxHalf;                     // [kTok][half]
    long long *slot = (long long *)(sn + kTok * kMaxHalf);  // element offset of (page, head 0) + 64 * slot
    const int *pos7 = (const int *)(slot + kTok);             // position % 8 of each token
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t0 = 0; t0 < c.n_valid; t0 += kTok) {
      const int nt = min(kTok, c.n_valid - t0);
      if (!(c.prepared && t0 == 0)) {
        __syncthreads();
        stage(c, extra, t0, nt, threadIdx.x, blockDim.x);
      }
      __syncthreads();
      const int nw = blockDim.x >> 5;
      for (int u = lane; u < units; u += 32) {
        const int hh = u >> pairs_log, j = 2 * (u & ((1 << pairs_log) - 1));
        const int f = hh * hd + j, fg = c.m0 + f;
        const int fh = fg - j;  // first feature of the head
        const bool rot = fg < qdim + kdim;
        bf16 *base_q = nullptr, *base_kv = nullptr;
        if (fh < qdim) {
          base_q = o.q + fh + j;
        } else {
          const bool is_k = fh < qdim + kdim;
          const int head = (fh - (is_k ? qdim : qdim + kdim)) / hd;
          base_kv = (is_k ? o.k_pool : o.v_pool) + (long long)head * o.pg * hd;
        }
        // four tokens per step: all shared-memory reads first, then math, then stores
        for (int tb = warp; tb < nt; tb += 4 * nw) {
          float a0[4], a1[4], b0[4], b1[4], c0[4], c1[4], s0[4], s1[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int t = min(tb + q * nw, nt - 1), tt = t0 + t;
            a0[q] = tile[f * ldc + (tt ^ (f & c.swz))];
            a1[q] = tile[(f + 1) * ldc + (tt ^ ((f + 1) & c.swz))];
            b0[q] = tile[(f + half) * ldc + (tt ^ ((f + half) & c.swz))];
            b1[q] = tile[(f + half + 1) * ldc + (tt ^ ((f + half + 1) & c.swz))];
            c0[q] = cs[t * half + j];
            c1[q] = cs[t * half + j + 1];
            s0[q] = sn[t * half + j];
            s1[q] = sn[t * half + j + 1];
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int t = tb + q * nw;
            if (t >= nt) break;
            float lo0 = a0[q], lo1 = a1[q], hi0 = b0[q], hi1 = b1[q];
            if (rot) {
              lo0 = a0[q] * c0[q] - b0[q] * s0[q];
              lo1 = a1[q] * c1[q] - b1[q] * s1[q];
              hi0 = b0[q] * c0[q] + a0[q] * s0[q];
              hi1 = b1[q] * c1[q] + a1[q] * s1[q];
            }
            if (base_q) {
              bf16 *dst = base_q + (size_t)(c.n0 + t0 + t) * qdim;
              *(__nv_bfloat162 *)dst = __floats2bfloat162_rn(lo0, lo1);
              *(__nv_bfloat162 *)(dst + half) = __floats2bfloat162_rn(hi0, hi1);
            } else {  // pool: feature f of slot s in sub-block f/64, chunk ((f%64)/8) ^ (s%8)
              const int s7 = pos7[t];
              bf16 *row = base_kv + slot[t];
              const int f0 = j, f1 = j + half;
              *(__nv_bfloat162 *)(row + (size_t)(f0 >> 6) * o.pg * 64 + ((((f0 & 63) >> 3) ^ s7) << 3) + (f0 & 7)) =
                  __floats2bfloat162_rn(lo0, lo1);
              *(__nv_bfloat162 *)(row + (size_t)(f1 >> 6) * o.pg * 64 + ((((f1 & 63) >> 3) ^ s7) << 3) + (f1 & 7)) =
                  __floats2bfloat162_rn(hi0, hi1);
            }
          }
        }
      }
    }
  }
};

// h[token][feature] += tile; lanes walk features (coalesced).  A warp takes
// 16 of its tokens x 4 feature groups of 32 at a time and issues all 64
// loads before any store.  Split-K with slices of up to kMaxW tokens:
// prepare() copies the slice's h rows into shared memory of their own right
// after the wait on the previous kernel, so their latency hides under the
// main loop.
struct EpiResidual {
  static constexpr int kMaxW = 64;
  static constexpr size_t extra_smem = 0;
  static constexpr bool kPrepEarly = false;  // h was written by earlier kernels
  static constexpr size_t prep_bytes(int w) { return w <= kMaxW ? (size_t)w * 128 * sizeof(float) : 0; }
  float *h;
  int ldh;
  // Split-K: feature row f of the slice gets its reduced sums v[j] for the
  // slice's tokens t0 + j straight from the reduction (lanes walk features:
  // one coalesced 128-byte store per token and warp); hb: the rows staged
  // by prepare(), or null.
  static constexpr bool kDirect = true;
  __device__ void direct(const TileCtx &c, int f, int t0, const float (&v)[32], unsigned char *pre) const {
    if (f >= c.m_valid) return;
    const float *hb = (const float *)pre;
    float *dst = h + (size_t)(c.n0 + t0) * ldh + c.m0 + f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int t = t0 + j;
      if (t < c.n_valid) {
        const float hv = hb ? hb[t * 128 + f] : dst[(size_t)j * ldh];
        dst[(size_t)j * ldh] = hv + v[j];
      }
    }
  }
  __device__ void prepare(const TileCtx &c, unsigned char *extra, int tid, int nthr) const {
    float4 *hb = (float4 *)extra;  // [token][128 features]
    const int n4 = min(c.n_valid, kMaxW) * 32;
    for (int i0 = 0; i0 < n4; i0 += nthr * 16) {
      float4 r[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = i0 + tid + nthr * u, t = i >> 5, f4 = i & 31;
        if (i < n4 && 4 * f4 < c.m_valid) r[u] = ((const float4 *)(h + (size_t)(c.n0 + t) * ldh + c.m0))[f4];
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = i0 + tid + nthr * u;
        if (i < n4 && 4 * (i & 31) < c.m_valid) hb[i] = r[u];
      }
    }
  }
  __device__ void operator()(float *tile, int ldc, const TileCtx &c, unsigned char *extra) const {
    const float *hb = c.prepared ? (const float *)extra : nullptr;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int f0 = 0; f0 < c.m_valid; f0 += 128) {
      for (int tb = warp; tb < c.n_valid; tb += 16 * nw) {
        float v[4][16];
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const int t = tb + u * nw, f = f0 + 32 * g + lane;
            v[g][u] = (f < c.m_valid && t < c.n_valid)
                          ? (hb ? hb[t * 128 + f] : h[(size_t)(c.n0 + t) * ldh + c.m0 + f])
                          : 0.0f;
          }
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const int t = tb + u * nw, f = f0 + 32 * g + lane;
            if (f < c.m_valid && t < c.n_valid)
              h[(size_t)(c.n0 + t) * ldh + c.m0 + f] = v[g][u] + tile[f * ldc + (t ^ (f & c.swz))];
          }
      }
    }
  }
};

TcArgs targs(int M, int N, int K, const bf16 *a, const bf16 *b, int *err, float *xchg = nullptr) {
  TcArgs g{};
  g.xchg = xchg;
  g.M = M;
  g.N = N;
  g.K = K;
  g.a = a;
  g.b = b;
  g.err = err;
  return g;
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    cudaGetLastError();
  }
  return fn;
}

cudaError_t make_tmap_bf16(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols,
                           uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  if (rows == 0) rows = 1;  // an empty operand still needs a valid map; nothing is read
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Encoded maps depend only on (address, shape, box); the decoder reuses the
// same weight and activation buffers every step, so each map is encoded once
// and copied into the launch parameters afterwards.
namespace {
struct TmapKey {
  const void *p;
  uint64_t rows, cols;
  uint32_t box;
  bool operator==(const TmapKey &o) const {
    return p == o.p && rows == o.rows && cols == o.cols && box == o.box;
  }
};
struct TmapKeyHash {
  size_t operator()(const TmapKey &k) const {
    size_t h = std::hash<const void *>()(k.p);
    h ^= std::hash<uint64_t>()(k.rows * 1000003ull + k.cols) + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
    return h ^ (k.box * 0x85ebca6bu);
  }
};
std::mutex g_tmap_mu;
std::unordered_map<TmapKey, CUtensorMap, TmapKeyHash> g_tmaps;
}  // namespace

static cudaError_t tmap_cached(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols,
                               uint32_t box) {
  const TmapKey key{ptr, rows, cols, box};
  std::lock_guard<std::mutex> lock(g_tmap_mu);
  auto it = g_tmaps.find(key);
  if (it != g_tmaps.end()) {
    *map = it->second;
    return cudaSuccess;
  }
  cudaError_t e = make_tmap_bf16(map, ptr, rows, cols, box);
  if (e != cudaSuccess) return e;
  if (g_tmaps.size() > 16384) g_tmaps.clear();
  g_tmaps.emplace(key, *map);
  return cudaSuccess;
}

cudaError_t tmap_bf16_cached(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols,
                             uint32_t box) {
  return tmap_cached(map, ptr, rows, cols, box);
}

// Projections: A = weights [M][K] (rows = output features), B = activations
// [T][K], both as operand tiles; the tile is [feature][token].

// Streaming multiprocessors of the current device (cached per device).
static int num_sms() {
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

// Clusters for a launch with a known number of output units: one CTA per SM
// at most, no more clusters than units.
static int plain_clusters(int units, int split) {
  int nc = num_sms() / split;
  if (nc > units) nc = units;
  return nc < 1 ? 1 : nc;
}

// Split for a plain projection: the largest of 4, 2, 1 that keeps at least
// two K tiles per split and every CTA resident at once.
static int pick_split(int units, int kt) {
  int s = 4;
  while (s > 1 && (kt < 2 * s || units * s > num_sms())) s >>= 1;
  return s;
}

template <class Epi>
static cudaError_t launch_split(const TcArgs &g,
                                const Epi &epi, int n_clusters, int split, cudaStream_t st) {
  switch (split) {
    case 4: return launch_tc_sk<4>(g, epi, n_clusters, st);
    case 2: return launch_tc_sk<2>(g, epi, n_clusters, st);
    default: return launch_tc_sk<1>(g, epi, n_clusters, st);
  }
}

size_t gemm_xchg_bytes() { return tc::split_k_xchg_bytes(num_sms()); }

cudaError_t gemm_qkv(const bf16 *x_tiles, const bf16 *wqkv, int T, int d, const QkvOut &o,
                     int *err, float *xchg, cudaStream_t st) {
  const int M = (o.Hq + 2 * o.Hkv) * o.hd;
  if (o.hd / 2 > EpiQkv::kMaxHalf || 128 % o.hd || d % 64) return cudaErrorInvalidValue;
  EpiQkv epi{o};
  const TcArgs g = targs(M, T, d, wqkv, x_tiles, err, xchg);
  const int units = ceil_div(M, 128) * ceil_div(T, tc::kSkBN);
  // a canvas step (32 units at the full width) splits K four ways; a prompt
  // chunk or a lockstep batch has units enough for every SM unsplit
  const int split = pick_split(units, d / tc::kBK);
  return launch_split(g, epi, plain_clusters(units, split), split, st);
}

cudaError_t gemm_residual(const bf16 *act_tiles, const bf16 *w, int T, int K, int N, float *h, int *err,
                          float *xchg, cudaStream_t st) {
  if (K % 64) return cudaErrorInvalidValue;
  EpiResidual epi{h, N};
  const int units = ceil_div(N, 128) * ceil_div(T, tc::kSkBN);
  const int split = pick_split(units, K / tc::kBK);
  return launch_split(targs(N, T, K, w, act_tiles, err, xchg), epi, plain_clusters(units, split), split, st);
}


// ---- failure detection -------------------------------------------------------
namespace {

// A wait that nothing completes: one thread initialises an mbarrier expecting
// one arrival that never comes and waits on it with the bounded wait every
// tensor-core kernel uses, which gives up after `limit` cycles, records code
// 99 in the error word and raises the CTA's abort flag.  Nothing is in flight.
__global__ void bounded_wait_selftest_kernel(int *err, long long limit) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    tc::mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    tc::mbar_wait(&bar, 0, err, 99, (volatile int *)&abort_flag, limit);
  }
}

}  // namespace

cudaError_t bounded_wait_selftest(int *err, long long limit_cycles, cudaStream_t st) {
  bounded_wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_cycles);
  return cudaGetLastError();
}

}  // namespace dg
