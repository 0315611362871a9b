// Warp-level bf16 tensor-core GEMM  D[M][N] = A[M][K] . B[N][K]^T  (fp32
// accumulation) with a cooperative epilogue on the fp32 tile in shared
// memory.  Both operands are K-contiguous (row-major weights [out][in] and
// activations [token][in]); B rows may be gathered through an index list and
// the launch may be "grouped" over experts through a device work list.
#pragma once
#include "common.cuh"

namespace dg {

struct GemmArgs {
  const bf16 *A;           // [M][lda] (+ group * a_group_stride)
  const bf16 *A2;          // optional second A ([M][lda]); D += A2 . B^T too (hi/lo split)
  long long lda;
  long long a_group_stride;
  const bf16 *B;           // rows b_row(n)
  long long ldb;
  const int *b_rows;       // gather list or null
  int M, N, K;
  // grouped launch: blockIdx.y indexes work items (group, n0); group g owns
  // B rows [group_offs[g], group_offs[g+1]) of the gather list / row space.
  const int *work;         // [n_work][2] or null
  const int *n_work;       // device count
  const int *group_offs;
};

// Context handed to the epilogue.
struct TileCtx {
  int m0, n0;      // tile origin in (M, N) of this group
  int m_valid;     // rows of the tile inside M
  int n_valid;     // columns of the tile inside the group's N
  int group;       // expert (0 if not grouped)
  int b_base;      // first B row of the group
};

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool pred) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  const int n = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void mma_bf16_16816(float *c, const uint32_t *a, const uint32_t *b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

template <int BM, int BN, int STAGES, int NA = 1>
struct GemmSmem {
  static constexpr int BK = 32;
  static constexpr int LDS = BK + 8;  // bf16 per staged row (80 B, conflict-free fragments)
  static constexpr int LDC = BN + 1;  // fp32 per epilogue row (odd: conflict-free columns)
  static constexpr size_t pipe = (size_t)STAGES * (NA * BM + BN) * LDS * sizeof(bf16);
  static constexpr size_t tile = (size_t)BM * LDC * sizeof(float);
  static constexpr size_t bytes = pipe > tile ? pipe : tile;
};

// Epi: struct with `static constexpr size_t extra_smem` and
//   __device__ void operator()(float *tile, int ldc, const TileCtx &, unsigned char *extra)
// NA = 2: A is given as two bf16 matrices whose sum is the operand (hi + lo
// split of an fp32 activation); both are multiplied with the same B tiles.
template <int BM, int BN, int WM, int WN, int STAGES, class Epi, int NA = 1>
__global__ void __launch_bounds__(WM *WN * 32) gemm_kernel(GemmArgs g, Epi epi) {
  using S = GemmSmem<BM, BN, STAGES, NA>;
  constexpr int NT = WM * WN * 32;
  constexpr int BK = S::BK, LDS = S::LDS;
  constexpr int TM = BM / WM, TN = BN / WN;
  constexpr int FM = TM / 16, FN = TN / 8;
  static_assert(TM % 16 == 0 && TN % 8 == 0, "warp tile");
  extern __shared__ __align__(16) unsigned char smem[];
  bf16 *As = (bf16 *)smem;                 // [STAGES][NA][BM][LDS]
  bf16 *Bs = As + STAGES * NA * BM * LDS;

  TileCtx ctx;
  ctx.m0 = blockIdx.x * BM;
  ctx.group = 0;
  ctx.b_base = 0;
  int n_total = g.N;
  if (g.work) {
    const int w = blockIdx.y;
    if (w >= *g.n_work) return;
    ctx.group = g.work[2 * w];
    ctx.n0 = g.work[2 * w + 1];
    ctx.b_base = g.group_offs[ctx.group];
    n_total = g.group_offs[ctx.group + 1] - ctx.b_base;
  } else {
    ctx.n0 = blockIdx.y * BN;
  }
  ctx.m_valid = min(BM, g.M - ctx.m0);
  ctx.n_valid = min(BN, n_total - ctx.n0);
  if (ctx.m_valid <= 0 || ctx.n_valid <= 0) return;
  const bf16 *A = g.A + (long long)ctx.group * g.a_group_stride;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp / WN, wn = warp % WN;
  const int KT = g.K / BK;

  auto load_stage = [&](int st, int kt) {
    const int k0 = kt * BK;
    bf16 *as = As + st * NA * BM * LDS;
    bf16 *bs = Bs + st * BN * LDS;
    for (int c = tid; c < NA * BM * 4; c += NT) {
      const int h = c / (BM * 4), cc = c % (BM * 4);
      const int r = cc >> 2, q = cc & 3;
      const bool ok = r < ctx.m_valid;
      const bf16 *base = (NA == 2 && h == 1) ? g.A2 : A;
      const bf16 *src = base + (long long)(ok ? ctx.m0 + r : 0) * g.lda + k0 + q * 8;
      cp_async16(as + (h * BM + r) * LDS + q * 8, src, ok);
    }
    for (int c = tid; c < BN * 4; c += NT) {
      const int r = c >> 2, q = c & 3;
      const bool ok = r < ctx.n_valid;
      long long row = 0;
      if (ok) {
        const int n = ctx.b_base + ctx.n0 + r;
        row = g.b_rows ? g.b_rows[n] : n;
      }
      cp_async16(bs + r * LDS + q * 8, g.B + row * g.ldb + k0 + q * 8, ok);
    }
  };

  float acc[FM][FN][4];
#pragma unroll
  for (int i = 0; i < FM; ++i)
#pragma unroll
    for (int j = 0; j < FN; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][j][r] = 0.0f;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < KT) load_stage(s, s);
    cp_async_commit();
  }
  for (int kt = 0; kt < KT; ++kt) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    const int nk = kt + STAGES - 1;
    if (nk < KT) load_stage(nk % STAGES, nk);
    cp_async_commit();
    const bf16 *as0 = As + (kt % STAGES) * NA * BM * LDS;
    const bf16 *bs = Bs + (kt % STAGES) * BN * LDS;
#pragma unroll
    for (int kk = 0; kk < BK; kk += 16) {
      uint32_t bfr[FN][2];
#pragma unroll
      for (int j = 0; j < FN; ++j) {
        const bf16 *p = bs + (wn * TN + j * 8 + (lane >> 2)) * LDS + kk + 2 * (lane & 3);
        bfr[j][0] = *(const uint32_t *)p;
        bfr[j][1] = *(const uint32_t *)(p + 8);
      }
#pragma unroll
      for (int h = 0; h < NA; ++h) {
        const bf16 *as = as0 + h * BM * LDS;
        uint32_t af[FM][4];
#pragma unroll
        for (int i = 0; i < FM; ++i) {
          const bf16 *p = as + (wm * TM + i * 16 + (lane >> 2)) * LDS + kk + 2 * (lane & 3);
          af[i][0] = *(const uint32_t *)p;
          af[i][1] = *(const uint32_t *)(p + 8 * LDS);
          af[i][2] = *(const uint32_t *)(p + 8);
          af[i][3] = *(const uint32_t *)(p + 8 * LDS + 8);
        }
#pragma unroll
        for (int i = 0; i < FM; ++i)
#pragma unroll
          for (int j = 0; j < FN; ++j) mma_bf16_16816(acc[i][j], af[i], bfr[j]);
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  float *tile = (float *)smem;
#pragma unroll
  for (int i = 0; i < FM; ++i)
#pragma unroll
    for (int j = 0; j < FN; ++j) {
      const int r = wm * TM + i * 16 + (lane >> 2);
      const int c = wn * TN + j * 8 + 2 * (lane & 3);
      tile[r * S::LDC + c] = acc[i][j][0];
      tile[r * S::LDC + c + 1] = acc[i][j][1];
      tile[(r + 8) * S::LDC + c] = acc[i][j][2];
      tile[(r + 8) * S::LDC + c + 1] = acc[i][j][3];
    }
  __syncthreads();
  epi(tile, S::LDC, ctx, smem + S::bytes);
}

template <int BM, int BN, int WM, int WN, int STAGES, class Epi, int NA = 1>
cudaError_t launch_gemm(const GemmArgs &g, const Epi &epi, int grid_y, cudaStream_t st) {
  using S = GemmSmem<BM, BN, STAGES, NA>;
  const size_t smem = S::bytes + Epi::extra_smem;
  auto kern = gemm_kernel<BM, BN, WM, WN, STAGES, Epi, NA>;
  static unsigned long long attr_set = 0;  // per device: one attribute call per instantiation
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !((attr_set >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set |= 1ull << dev;
  }
  if (grid_y <= 0) return cudaSuccess;
  dim3 grid(ceil_div(g.M, BM), grid_y);
  kern<<<grid, WM * WN * 32, smem, st>>>(g, epi);
  return cudaGetLastError();
}

}  // namespace dg
