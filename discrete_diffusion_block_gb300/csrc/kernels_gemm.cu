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
#include "sampler.cuh"

namespace dg {

namespace {

// q/k/v projection: RoPE (rotate-half pairs (j, j+hd/2)) on q and k at
// absolute position pos0 + token; q to [T][Hq*hd]; k and v straight into the
// paged pool slice of this layer.  The tile's tokens' cos/sin rows and page
// slots are first staged in shared memory, so the element loop only reads
// shared memory and issues stores.
template <int BN>
struct EpiQkv {
  static constexpr int kMaxHalf = 64;
  static constexpr size_t extra_smem = (size_t)BN * kMaxHalf * 2 * sizeof(float) + BN * sizeof(long long);
  QkvOut o;
  __device__ void operator()(float *tile, int ldc, const TileCtx &c, unsigned char *extra) const {
    const int BM = c.m_valid;
    const int half = o.hd / 2, qdim = o.Hq * o.hd, kdim = o.Hkv * o.hd;
    float *cs = (float *)extra;                  // [BN][half]
    float *sn = cs + BN * kMaxHalf;              // [BN][half]
    long long *slot = (long long *)(sn + BN * kMaxHalf);  // element offset of (page, 0, slot, 0)
    for (int i = threadIdx.x; i < c.n_valid * half; i += blockDim.x) {
      const int t = i / half, j = i % half;
      const size_t p = (size_t)(o.pos0 + c.n0 + t);
      cs[t * half + j] = o.cos_t[p * half + j];
      sn[t * half + j] = o.sin_t[p * half + j];
    }
    for (int t = threadIdx.x; t < c.n_valid; t += blockDim.x) {
      const int p = o.pos0 + c.n0 + t;
      slot[t] = ((long long)o.page_table[p / o.pg] * o.Hkv * o.pg + p % o.pg) * o.hd;
    }
    __syncthreads();
#pragma unroll 4
    for (int idx = threadIdx.x; idx < c.n_valid * BM; idx += blockDim.x) {
      const int t = idx / BM, f = idx % BM;
      const int fg = c.m0 + f;
      const int tok = c.n0 + t;
      const int j = fg % o.hd;
      float val;
      if (fg < qdim + kdim) {
        const int jj = j % half;
        const float cv = cs[t * half + jj], sv = sn[t * half + jj];
        val = j < half ? tile[f * ldc + t] * cv - tile[(f + half) * ldc + t] * sv
                       : tile[(f - half) * ldc + t] * sv + tile[f * ldc + t] * cv;
      } else {
        val = tile[f * ldc + t];
      }
      const bf16 b = __float2bfloat16_rn(val);
      if (fg < qdim) {
        o.q[(size_t)tok * qdim + fg] = b;
      } else {
        const bool is_k = fg < qdim + kdim;
        const int head = (fg - (is_k ? qdim : qdim + kdim)) / o.hd;
        (is_k ? o.k_pool : o.v_pool)[slot[t] + (long long)head * o.pg * o.hd + j] = b;
      }
    }
  }
};

// h[token][feature] += tile; eight independent loads in flight per thread.
struct EpiResidual {
  static constexpr size_t extra_smem = 0;
  float *h;
  int ldh;
  __device__ void operator()(float *tile, int ldc, const TileCtx &c, unsigned char *) const {
    const int n = c.n_valid * c.m_valid;
    for (int base = threadIdx.x; base < n; base += 8 * blockDim.x) {
      float v[8];
      size_t off[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int idx = base + u * blockDim.x;
        const int t = idx / c.m_valid, f = idx % c.m_valid;
        off[u] = (size_t)(c.n0 + t) * ldh + c.m0 + f;
        v[u] = idx < n ? h[off[u]] : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int idx = base + u * blockDim.x;
        if (idx < n) {
          const int t = idx / c.m_valid, f = idx % c.m_valid;
          h[off[u]] = v[u] + tile[f * ldc + t];
        }
      }
    }
  }
};

// out[token][feature] = tile (grouped launches address rows from b_base)
struct EpiStore {
  static constexpr size_t extra_smem = 0;
  float *out;
  int ldo;
  __device__ void operator()(float *tile, int ldc, const TileCtx &c, unsigned char *) const {
    for (int idx = threadIdx.x; idx < c.n_valid * c.m_valid; idx += blockDim.x) {
      const int t = idx / c.m_valid, f = idx % c.m_valid;
      out[(size_t)(c.b_base + c.n0 + t) * ldo + c.m0 + f] = tile[f * ldc + t];
    }
  }
};

// SwiGLU on a 128-row tile holding 64 gate rows then the matching 64 up rows.
struct EpiSwiGlu {
  static constexpr size_t extra_smem = 0;
  bf16 *act;
  int F;
  __device__ void operator()(float *tile, int ldc, const TileCtx &c, unsigned char *) const {
    const int fb = c.m0 / 128;
    for (int idx = threadIdx.x; idx < c.n_valid * 64; idx += blockDim.x) {
      const int t = idx / 64, j = idx % 64;
      const float g = tile[j * ldc + t], u = tile[(64 + j) * ldc + t];
      act[(size_t)(c.b_base + c.n0 + t) * F + fb * 64 + j] = __float2bfloat16_rn(silu_f(g) * u);
    }
  }
};

// LM head: the tile is [token][256 vocab]; reduce it to sampler partials.
template <int BM>
struct EpiLmHead {
  static constexpr size_t extra_smem = (size_t)BM * (kVocabTile + 1) * sizeof(float) + BM * 8;
  PartialPlanes P;
  int tiles;
  uint32_t ctr2, key0, key1;
  const StepParams *dyn;  // when set, the stream words come from device memory
  __device__ void operator()(float *tile, int ldc, const TileCtx &c, unsigned char *extra) const {
    PartialScratch sc;
    sc.kap = (float *)extra;
    sc.rm = sc.kap + BM * ldc;
    sc.ra = (int *)(sc.rm + BM);
    const uint32_t c2 = dyn ? dyn->ctr2 : ctr2, k0 = dyn ? dyn->key0 : key0, k1 = dyn ? dyn->key1 : key1;
    block_tile_partials(tile, ldc, sc, c.m_valid, c.n0, c.n0 / kVocabTile, tiles, c.m0, c2, k0, k1,
                        P, c.m0);
  }
};

// out[row][col] = tile, rows = tokens (A operand), cols = vocab (B operand).
struct EpiStoreRows {
  static constexpr size_t extra_smem = 0;
  float *out;
  long long ldo;
  __device__ void operator()(float *tile, int ldc, const TileCtx &c, unsigned char *) const {
    for (int idx = threadIdx.x; idx < c.m_valid * c.n_valid; idx += blockDim.x) {
      const int r = idx / c.n_valid, col = idx % c.n_valid;
      out[(size_t)(c.m0 + r) * ldo + c.n0 + col] = tile[r * ldc + col];
    }
  }
};

TcArgs targs(int M, int N, int K, int *err) {
  TcArgs g{};
  g.M = M;
  g.N = N;
  g.K = K;
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

#define TMAP(map, ptr, rows, cols, box)                                            \
  do {                                                                             \
    cudaError_t e_ = tmap_cached(&(map), (ptr), (rows), (cols), (box));            \
    if (e_ != cudaSuccess) return e_;                                              \
  } while (0)

// Projections: A = weights [M][K] (rows = output features), B = activations
// [T][K]; the tile is [feature][token].
cudaError_t gemm_qkv(const bf16 *xn, const bf16 *wqkv, int T, int d, const QkvOut &o,
                     int *err, cudaStream_t st) {
  const int M = (o.Hq + 2 * o.Hkv) * o.hd;
  CUtensorMap ta, tb;
  TMAP(ta, wqkv, M, d, 128);
  TMAP(tb, xn, T, d, 64);
  if (o.hd / 2 > EpiQkv<64>::kMaxHalf) return cudaErrorInvalidValue;
  EpiQkv<64> epi{o};
  return launch_tc<64, 4, 1, 128>(ta, ta, tb, targs(M, T, d, err), epi, ceil_div(T, 64), st);
}

cudaError_t gemm_residual(const bf16 *act, const bf16 *w, int T, int K, int N, float *h, int *err,
                          cudaStream_t st) {
  CUtensorMap ta, tb;
  TMAP(ta, w, N, K, 128);
  TMAP(tb, act, T, K, 64);
  EpiResidual epi{h, N};
  return launch_tc<64, 4, 1, 128>(ta, ta, tb, targs(N, T, K, err), epi, ceil_div(T, 64), st);
}

cudaError_t gemm_store_f32(const bf16 *act, const bf16 *w, int T, int K, int N, float *out, int *err,
                           cudaStream_t st) {
  CUtensorMap ta, tb;
  TMAP(ta, w, N, K, 128);
  TMAP(tb, act, T, K, 64);
  EpiStore epi{out, N};
  return launch_tc<64, 4, 1, 128>(ta, ta, tb, targs(N, T, K, err), epi, ceil_div(T, 64), st);
}

// Experts: A = the expert's weight rows (2-D view over all experts), B = the
// expert's routed rows, packed contiguously in expert order.
cudaError_t gemm_expert_gate_up(const bf16 *x_perm, int rows, const bf16 *wgu, const int *offs,
                                const int *work, const int *n_work, int max_work, int E, int d,
                                int F, bf16 *act, int *err, cudaStream_t st) {
  CUtensorMap ta, tb;
  TMAP(ta, wgu, (uint64_t)E * 2 * F, d, 128);
  TMAP(tb, x_perm, rows, d, kExpertTileRows);
  TcArgs g = targs(2 * F, 0, d, err);
  g.a_group_rows = 2 * F;
  g.work = work;
  g.n_work = n_work;
  g.group_offs = offs;
  EpiSwiGlu epi{act, F};
  return launch_tc<kExpertTileRows, 4, 1, 128>(ta, ta, tb, g, epi, max_work, st);
}

cudaError_t gemm_expert_down(const bf16 *act, int rows, const bf16 *wd, const int *offs,
                             const int *work, const int *n_work, int max_work, int E, int d, int F,
                             float *y, int *err, cudaStream_t st) {
  CUtensorMap ta, tb;
  TMAP(ta, wd, (uint64_t)E * d, F, 128);
  TMAP(tb, act, rows, F, kExpertTileRows);
  TcArgs g = targs(d, 0, F, err);
  g.a_group_rows = d;
  g.work = work;
  g.n_work = n_work;
  g.group_offs = offs;
  EpiStore epi{y, d};
  return launch_tc<kExpertTileRows, 4, 1, 128>(ta, ta, tb, g, epi, max_work, st);
}

// LM head: A = normalised token rows (hi, and lo of a hi/lo split), B = the
// vocab rows of W_out, one 256-wide vocab tile per CTA column.
cudaError_t gemm_lm_head_partials(const bf16 *xn, const bf16 *xn_lo, const bf16 *w_out, int T, int d,
                                  int V, uint64_t seed, int canvas, int step, void *partials,
                                  int *err, cudaStream_t st, const StepParams *dyn) {
  CUtensorMap ta, ta2, tb;
  TMAP(ta, xn, T, d, 128);
  TMAP(ta2, xn_lo ? xn_lo : xn, T, d, 128);
  TMAP(tb, w_out, V, d, 256);
  EpiLmHead<64> epi;
  epi.tiles = V / kVocabTile;
  epi.P = PartialPlanes::at(partials, T, epi.tiles);
  epi.ctr2 = gumbel_ctr2(canvas, step);
  epi.key0 = (uint32_t)seed;
  epi.key1 = (uint32_t)(seed >> 32);
  epi.dyn = dyn;
  const TcArgs g = targs(T, V, d, err);
  if (xn_lo) return launch_tc<256, 3, 2, 64>(ta, ta2, tb, g, epi, V / kVocabTile, st);
  return launch_tc<256, 4, 1, 64>(ta, ta, tb, g, epi, V / kVocabTile, st);
}

cudaError_t gemm_lm_head_logits(const bf16 *xn, const bf16 *xn_lo, const bf16 *w_out, int T, int d,
                                int V, float *logits, int *err, cudaStream_t st) {
  CUtensorMap ta, ta2, tb;
  TMAP(ta, xn, T, d, 128);
  TMAP(ta2, xn_lo ? xn_lo : xn, T, d, 128);
  TMAP(tb, w_out, V, d, 256);
  EpiStoreRows epi{logits, V};
  const TcArgs g = targs(T, V, d, err);
  if (xn_lo) return launch_tc<256, 3, 2, 64>(ta, ta2, tb, g, epi, V / kVocabTile, st);
  return launch_tc<256, 4, 1, 64>(ta, ta, tb, g, epi, V / kVocabTile, st);
}

}  // namespace dg
