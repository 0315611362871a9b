// Projection, expert and LM-head GEMMs of the decoder with their fused
// epilogues.  Weights are the A operand (rows = output features) for every
// projection (the token count is the short side), except the LM head whose
// epilogue needs a token's whole 256-wide vocab tile in one row.
#include "gemm_mma.cuh"
#include "internal.h"
#include "sampler.cuh"

namespace dg {

namespace {

// q/k/v projection: RoPE (rotate-half pairs (j, j+hd/2)) on q and k at
// absolute position pos0 + token; q to [T][Hq*hd]; k and v straight into the
// paged pool slice of this layer.
struct EpiQkv {
  static constexpr size_t extra_smem = 0;
  QkvOut o;
  __device__ void operator()(float *tile, int ldc, const TileCtx &c, unsigned char *) const {
    const int BM = c.m_valid;
    const int half = o.hd / 2, qdim = o.Hq * o.hd, kdim = o.Hkv * o.hd;
    for (int idx = threadIdx.x; idx < c.n_valid * BM; idx += blockDim.x) {
      const int t = idx / BM, f = idx % BM;
      const int fg = c.m0 + f;
      const int tok = c.n0 + t;
      const int p = o.pos0 + tok;
      const int j = fg % o.hd;
      float val;
      if (fg < qdim + kdim) {
        const int jj = j % half;
        const float cs = o.cos_t[(size_t)p * half + jj], sn = o.sin_t[(size_t)p * half + jj];
        if (j < half) {
          val = tile[f * ldc + t] * cs - tile[(f + half) * ldc + t] * sn;
        } else {
          val = tile[(f - half) * ldc + t] * sn + tile[f * ldc + t] * cs;
        }
      } else {
        val = tile[f * ldc + t];
      }
      const bf16 b = __float2bfloat16_rn(val);
      if (fg < qdim) {
        o.q[(size_t)tok * qdim + fg] = b;
      } else {
        const bool is_k = fg < qdim + kdim;
        const int head = (fg - (is_k ? qdim : qdim + kdim)) / o.hd;
        const size_t dst =
            (((size_t)o.page_table[p / o.pg] * o.Hkv + head) * o.pg + p % o.pg) * o.hd + j;
        (is_k ? o.k_pool : o.v_pool)[dst] = b;
      }
    }
  }
};

// h[token][feature] += tile
struct EpiResidual {
  static constexpr size_t extra_smem = 0;
  float *h;
  int ldh;
  __device__ void operator()(float *tile, int ldc, const TileCtx &c, unsigned char *) const {
    for (int idx = threadIdx.x; idx < c.n_valid * c.m_valid; idx += blockDim.x) {
      const int t = idx / c.m_valid, f = idx % c.m_valid;
      h[(size_t)(c.n0 + t) * ldh + c.m0 + f] += tile[f * ldc + t];
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
  __device__ void operator()(float *tile, int ldc, const TileCtx &c, unsigned char *extra) const {
    PartialScratch sc;
    sc.kap = (float *)extra;
    sc.rm = sc.kap + BM * ldc;
    sc.ra = (int *)(sc.rm + BM);
    block_tile_partials(tile, ldc, sc, c.m_valid, c.n0, c.n0 / kVocabTile, tiles, c.m0, ctr2, key0,
                        key1, P, c.m0);
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

GemmArgs plain(const bf16 *A, long long lda, const bf16 *B, long long ldb, int M, int N, int K) {
  GemmArgs g{};
  g.A = A;
  g.lda = lda;
  g.B = B;
  g.ldb = ldb;
  g.M = M;
  g.N = N;
  g.K = K;
  return g;
}

}  // namespace

cudaError_t gemm_qkv(const bf16 *xn, const bf16 *wqkv, int T, int d, const QkvOut &o,
                     cudaStream_t st) {
  const int M = (o.Hq + 2 * o.Hkv) * o.hd;
  GemmArgs g = plain(wqkv, d, xn, d, M, T, d);
  EpiQkv epi{o};
  return launch_gemm<128, 64, 4, 2, 3>(g, epi, ceil_div(T, 64), st);
}

cudaError_t gemm_residual(const bf16 *act, const bf16 *w, int T, int K, int N, float *h,
                          cudaStream_t st) {
  GemmArgs g = plain(w, K, act, K, N, T, K);
  EpiResidual epi{h, N};
  return launch_gemm<128, 64, 4, 2, 3>(g, epi, ceil_div(T, 64), st);
}

cudaError_t gemm_store_f32(const bf16 *act, const bf16 *w, int T, int K, int N, float *out,
                           cudaStream_t st) {
  GemmArgs g = plain(w, K, act, K, N, T, K);
  EpiStore epi{out, N};
  return launch_gemm<128, 64, 4, 2, 3>(g, epi, ceil_div(T, 64), st);
}

cudaError_t gemm_expert_gate_up(const bf16 *xn, const bf16 *wgu, const int *perm_tok,
                                const int *offs, const int *work, const int *n_work, int max_work,
                                int d, int F, bf16 *act, cudaStream_t st) {
  GemmArgs g = plain(wgu, d, xn, d, 2 * F, 0, d);
  g.a_group_stride = (long long)2 * F * d;
  g.b_rows = perm_tok;
  g.work = work;
  g.n_work = n_work;
  g.group_offs = offs;
  EpiSwiGlu epi{act, F};
  return launch_gemm<128, kExpertTileRows, 4, 2, 3>(g, epi, max_work, st);
}

cudaError_t gemm_expert_down(const bf16 *act, const bf16 *wd, const int *offs, const int *work,
                             const int *n_work, int max_work, int d, int F, float *y,
                             cudaStream_t st) {
  GemmArgs g = plain(wd, F, act, F, d, 0, F);
  g.a_group_stride = (long long)d * F;
  g.work = work;
  g.n_work = n_work;
  g.group_offs = offs;
  EpiStore epi{y, d};
  return launch_gemm<128, kExpertTileRows, 4, 2, 3>(g, epi, max_work, st);
}

cudaError_t gemm_lm_head_partials(const bf16 *xn, const bf16 *xn_lo, const bf16 *w_out, int T, int d,
                                  int V, uint64_t seed, int canvas, int step, void *partials,
                                  cudaStream_t st) {
  constexpr int BM = 64;
  GemmArgs g = plain(xn, d, w_out, d, T, V, d);
  g.A2 = xn_lo;
  EpiLmHead<BM> epi;
  epi.tiles = V / kVocabTile;
  epi.P = PartialPlanes::at(partials, T, epi.tiles);
  epi.ctr2 = gumbel_ctr2(canvas, step);
  epi.key0 = (uint32_t)seed;
  epi.key1 = (uint32_t)(seed >> 32);
  if (xn_lo) return launch_gemm<BM, kVocabTile, 2, 4, 3, EpiLmHead<BM>, 2>(g, epi, V / kVocabTile, st);
  return launch_gemm<BM, kVocabTile, 2, 4, 3>(g, epi, V / kVocabTile, st);
}

cudaError_t gemm_lm_head_logits(const bf16 *xn, const bf16 *xn_lo, const bf16 *w_out, int T, int d,
                                int V, float *logits, cudaStream_t st) {
  constexpr int BM = 64;
  GemmArgs g = plain(xn, d, w_out, d, T, V, d);
  g.A2 = xn_lo;
  EpiStoreRows epi{logits, V};
  if (xn_lo) return launch_gemm<BM, kVocabTile, 2, 4, 3, EpiStoreRows, 2>(g, epi, V / kVocabTile, st);
  return launch_gemm<BM, kVocabTile, 2, 4, 3>(g, epi, V / kVocabTile, st);
}

}  // namespace dg
