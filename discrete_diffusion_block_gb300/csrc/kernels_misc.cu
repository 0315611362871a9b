// Small kernels of the decoder: seeded weights, canvas initialisation,
// embedding gather, RMSNorm, RoPE tables, MoE routing / permutation /
// combination, KV append.
#include <math.h>
#include <stdlib.h>

#include "internal.h"

namespace dg {

namespace {

inline int grid_for(size_t n, int threads, int cap = 152 * 32) {
  size_t b = (n + threads - 1) / threads;
  if (b < 1) b = 1;
  return (int)(b < (size_t)cap ? b : (size_t)cap);
}

// ---- seeded synthetic weights ---------------------------------------------
// element e of tensor `tid`: Irwin-Hall(4) over one Philox4x32-10 call at
// counter (e mod 2^32, e div 2^32, tid, 1), scaled to the requested std and
// rounded to bf16.
__device__ __forceinline__ bf16 weight_element(uint64_t e, uint32_t tid, uint32_t k0, uint32_t k1,
                                               float scale) {
  const U4 w = philox10((uint32_t)e, (uint32_t)(e >> 32), tid, kTagWeight, k0, k1);
  const int s = (int)(w.w[0] >> 9) + (int)(w.w[1] >> 9) + (int)(w.w[2] >> 9) + (int)(w.w[3] >> 9);
  return __float2bfloat16_rn(__fmul_rn((float)(s - (1 << 24)), scale));
}

__global__ void fill_weights_kernel(bf16 *dst, uint64_t n, uint32_t k0, uint32_t k1, uint32_t tid,
                                    uint64_t e0, float scale) {
  for (uint64_t j = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; j < n;
       j += (uint64_t)gridDim.x * blockDim.x)
    dst[j] = weight_element(e0 + j, tid, k0, k1, scale);
}

// Expert weights are stored as operand tiles: a matrix with 128-row blocks
// and K-tiles of 64 columns is laid out [row block][k-tile][128][64], each
// 16 KB tile in the shared-memory order the tensor core reads (row r's
// 16-byte chunk c at chunk position c ^ (r % 8)), so that one contiguous bulk
// copy moves a tile.  Physical element p of a tile: row r = p / 64, logical
// column 8 ((p / 8 % 8) ^ (r % 8)) + p % 8 of the tile.
__device__ __forceinline__ void tile_coords(uint64_t j, int KT, uint64_t *blk, int *kt, int *r, int *c) {
  const int p = (int)(j & 8191);
  const uint64_t t = j >> 13;
  *kt = (int)(t % KT);
  *blk = t / KT;
  *r = p >> 6;
  *c = *kt * 64 + ((((p >> 3) & 7) ^ (*r & 7)) << 3) + (p & 7);
}

// Inverse of tiled_index: the (row, column) of element j of the operand tiles
// of a [rows][cols] matrix.
__device__ __forceinline__ void tiled_coords(int rows, int cols, uint64_t j, int *r, int *c) {
  const int b = (int)(j / ((uint64_t)128 * cols));
  const int rows_b = min(128, rows - 128 * b);
  const uint64_t within = j - (uint64_t)b * 128 * cols;
  const int kt = (int)(within / ((uint64_t)rows_b * 64));
  const int p = (int)(within - (uint64_t)kt * rows_b * 64);
  const int rr = p >> 6;
  *r = 128 * b + rr;
  *c = kt * 64 + ((((p >> 3) & 7) ^ (rr & 7)) << 3) + (p & 7);
}

// W_gate and W_up (logical [E][F][d] each): per expert, the operand tiles of
// W_gate,e ([F][d], tiled_index) followed by the operand tiles of W_up,e.
__global__ void fill_gate_up_kernel(bf16 *dst, int E, int F, int d, uint32_t k0, uint32_t k1,
                                    uint32_t tid_gate, uint32_t tid_up, float scale) {
  const uint64_t n = (uint64_t)E * 2 * F * d, per = (uint64_t)F * d;
  for (uint64_t j = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; j < n;
       j += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t mat = j / per;  // 2 e (gate) or 2 e + 1 (up)
    int r, c;
    tiled_coords(F, d, j - mat * per, &r, &c);
    const uint64_t logical = ((mat >> 1) * F + r) * d + c;
    dst[j] = weight_element(logical, (mat & 1) ? tid_up : tid_gate, k0, k1, scale);
  }
}

// A weight matrix [rows][cols] stored as operand tiles whose logical rows come
// from up to three generated tensors: rows [0, r1) of tensor tid0, [r1, r2)
// of tid1, [r2, rows) of tid2 (each row-major with `cols` columns).
__global__ void fill_tiled_kernel(bf16 *dst, int rows, int cols, int r1, int r2, uint32_t tid0, uint32_t tid1,
                                  uint32_t tid2, uint32_t k0, uint32_t k1, float scale) {
  const uint64_t n = (uint64_t)rows * cols;
  for (uint64_t j = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; j < n;
       j += (uint64_t)gridDim.x * blockDim.x) {
    int r, c;
    tiled_coords(rows, cols, j, &r, &c);
    const uint32_t tid = r < r1 ? tid0 : r < r2 ? tid1 : tid2;
    const int r0 = r < r1 ? 0 : r < r2 ? r1 : r2;
    dst[j] = weight_element((uint64_t)(r - r0) * cols + c, tid, k0, k1, scale);
  }
}

// W_down (logical [E][d][F]) as tiles of 128-row blocks, K = F.
__global__ void fill_down_kernel(bf16 *dst, int E, int F, int d, uint32_t k0, uint32_t k1, uint32_t tid,
                                 float scale) {
  const uint64_t n = (uint64_t)E * d * F;
  const int KT = F / 64, mB = d / 128;
  for (uint64_t j = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; j < n;
       j += (uint64_t)gridDim.x * blockDim.x) {
    uint64_t blk;
    int kt, r, c;
    tile_coords(j, KT, &blk, &kt, &r, &c);
    const int mb = (int)(blk % mB), e = (int)(blk / mB);
    const uint64_t logical = ((uint64_t)e * d + mb * 128 + r) * F + c;
    dst[j] = weight_element(logical, tid, k0, k1, scale);
  }
}

__global__ void fill_const_kernel(float *dst, size_t n, float v) {
  for (size_t j = blockIdx.x * (size_t)blockDim.x + threadIdx.x; j < n;
       j += (size_t)gridDim.x * blockDim.x)
    dst[j] = v;
}

// cos/sin of pos * base^(-2j/hd), evaluated in double, stored fp32.
__global__ void rope_table_kernel(float *ct, float *stt, int max_pos, int half, int hd,
                                  double base) {
  const size_t n = (size_t)max_pos * half;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int p = (int)(i / half), j = (int)(i % half);
    const double th = pow(base, -2.0 * j / hd);
    double s, c;
    sincos((double)p * th, &s, &c);
    ct[i] = (float)c;
    stt[i] = (float)s;
  }
}

// x_1 ~ Unif(V^C): id = floor(word0 * V / 2^32), word0 of Philox at (i, 0, k, 2).
// Request b (blockIdx.y) of a lockstep batch draws with sample seed + b.
__global__ void canvas_init_kernel(int *x, uint8_t *committed, int *last, int *stable, int C, int V,
                                   uint64_t seed, int canvas) {
  pdl_wait();
  pdl_trigger();
  const int p = blockIdx.x * blockDim.x + threadIdx.x, b = blockIdx.y, i = b * C + p;
  if (p >= C) return;
  const uint64_t s = seed + (uint64_t)b;
  const U4 w = philox10((uint32_t)p, 0u, (uint32_t)canvas, kTagInit, (uint32_t)s, (uint32_t)(s >> 32));
  x[i] = (int)(((uint64_t)w.w[0] * (uint64_t)V) >> 32);
  committed[i] = 0;
  last[i] = -1;
  stable[i] = 0;
}

__global__ void embed_kernel(float *h, const bf16 *table, const int *ids, int d) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const bf16 *row = table + (size_t)ids[t] * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) h[(size_t)t * d + c] = __bfloat162float(row[c]);
}

// y = x / sqrt(mean(x^2) + eps) * g, fp32 statistics, bf16 output; with
// out_lo the residual y - bf16(y) is stored too (hi + lo carries y to ~16 bits).
// One 128-thread block per row; the row is read once as float4 into
// registers (d <= 4096; longer rows are read twice).
constexpr int kNormThreads = 128, kNormVec = 8;
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(bf16 *out, bf16 *out_lo, const float *h,
                                                               const float *g, int d, float eps, int tiled_rows) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x, d4 = d >> 2;
  const float4 *x = (const float4 *)(h + (size_t)t * d);
  const float4 *g4 = (const float4 *)g;
  float4 v[kNormVec];
  float ss = 0.0f;
#pragma unroll
  for (int u = 0; u < kNormVec; ++u) {
    const int c = threadIdx.x + u * kNormThreads;
    v[u] = c < d4 ? x[c] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int u = 0; u < kNormVec; ++u) ss += v[u].x * v[u].x + v[u].y * v[u].y + v[u].z * v[u].z + v[u].w * v[u].w;
  for (int c = threadIdx.x + kNormVec * kNormThreads; c < d4; c += kNormThreads) {
    const float4 a = x[c];
    ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w;
  }
  __shared__ float red[kNormThreads / 32];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
  const float inv = rsqrtf(tot / d + eps);
  __nv_bfloat162 *o2 = (__nv_bfloat162 *)(out + (size_t)t * d);
  __nv_bfloat162 *l2 = out_lo ? (__nv_bfloat162 *)(out_lo + (size_t)t * d) : nullptr;
  for (int c = threadIdx.x, u = 0; c < d4; c += kNormThreads, ++u) {
    float4 a;
    if (u < kNormVec) {
#pragma unroll
      for (int q = 0; q < kNormVec; ++q)
        if (q == u) a = v[q];
    } else {
      a = x[c];
    }
    const float4 gg = g4[c];
    const float y0 = a.x * inv * gg.x, y1 = a.y * inv * gg.y, y2 = a.z * inv * gg.z, y3 = a.w * inv * gg.w;
    const __nv_bfloat162 h01 = __floats2bfloat162_rn(y0, y1), h23 = __floats2bfloat162_rn(y2, y3);
    if (tiled_rows > 0) {  // a tensor-core operand: operand tiles
      *(uint2 *)(out + tiled_index(tiled_rows, d, t, 4 * c)) =
          make_uint2(*(const uint32_t *)&h01, *(const uint32_t *)&h23);
    } else {
      o2[2 * c] = h01;
      o2[2 * c + 1] = h23;
    }
    if (out_lo) {
      const __nv_bfloat162 l01 = __floats2bfloat162_rn(y0 - __low2float(h01), y1 - __high2float(h01));
      const __nv_bfloat162 l23 = __floats2bfloat162_rn(y2 - __low2float(h23), y3 - __high2float(h23));
      if (tiled_rows > 0) {
        *(uint2 *)(out_lo + tiled_index(tiled_rows, d, t, 4 * c)) =
            make_uint2(*(const uint32_t *)&l01, *(const uint32_t *)&l23);
      } else {
        l2[2 * c] = l01;
        l2[2 * c + 1] = l23;
      }
    }
  }
}

// top-k of E router logits per token (value desc, expert id asc), softmax
// gates over the selected logits.  One warp per token, E <= 256, k <= 16.
// An unordered logit (NaN) never wins a comparison but a still-unselected
// expert is always taken over none, so every emitted id is in [0, E).

// Four bf16 values (one 8-byte load) to floats.
__device__ __forceinline__ float4 bf16x4_to_float4(uint2 w) {
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u), __uint_as_float(w.y << 16),
                     __uint_as_float(w.y & 0xffff0000u));
}

// h[t] (+)= sum_s gate[t][s] * y[slot_row[t*k+s]] (y bf16), slots in
// ascending order.  The token's gates and rows are staged first; each
// thread then has all k row loads of its 4-column group in flight at once.
__global__ void __launch_bounds__(256) combine_kernel(float4 *h, const uint2 *y, const float *gates,
                                                      const int *slot_row, int k, int d4,
                                                      int accumulate) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  __shared__ float g_s[16];
  __shared__ int r_s[16];
  if (threadIdx.x < k) {
    g_s[threadIdx.x] = gates[(size_t)t * k + threadIdx.x];
    r_s[threadIdx.x] = slot_row[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  for (int c = threadIdx.x; c < d4; c += blockDim.x) {
    uint2 v[16];
#pragma unroll
    for (int s = 0; s < 16; ++s)
      if (s < k) v[s] = y[(size_t)r_s[s] * d4 + c];
    float4 acc = accumulate ? h[(size_t)t * d4 + c] : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 mo = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < 16; ++s)
      if (s < k) {
        const float4 f = bf16x4_to_float4(v[s]);
        mo.x += g_s[s] * f.x;
        mo.y += g_s[s] * f.y;
        mo.z += g_s[s] * f.z;
        mo.w += g_s[s] * f.w;
      }
    h[(size_t)t * d4 + c] = make_float4(acc.x + mo.x, acc.y + mo.y, acc.z + mo.z, acc.w + mo.w);
  }
}

// combine_kernel followed by the RMSNorm of the updated row (the next
// layer's input norm, same formula as rmsnorm_kernel): one block per token,
// one 4-column group per thread (d4 <= 1024), so that the h row and eight
// expert rows of a column are in flight at once; the row stays in registers
// between the two steps.
__global__ void __launch_bounds__(1024, 2) combine_norm_kernel(float4 *h, const uint2 *y, const float *gates,
                                                            const int *slot_row, int k, int d4,
                                                            const float *gain, float eps, bf16 *x_tiles, int T) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x, c = threadIdx.x;
  const bool ok = c < d4;
  __shared__ float g_s[16];
  __shared__ int r_s[16];
  __shared__ float red[32];
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 acc = ok ? h[(size_t)t * d4 + c] : zero;
  if (threadIdx.x < k) {
    g_s[threadIdx.x] = gates[(size_t)t * k + threadIdx.x];
    r_s[threadIdx.x] = slot_row[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  float4 hv = zero;
  float ss = 0.0f;
  if (ok) {
    float4 mo = acc;  // h, then the gate-weighted expert rows in slot order
    for (int s0 = 0; s0 < k; s0 += 8) {  // eight expert rows in flight at a time, summed in slot order
      uint2 v[8];
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if (s0 + s < k) v[s] = y[(size_t)r_s[s0 + s] * d4 + c];
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if (s0 + s < k) {
          const float gs = g_s[s0 + s];
          const float4 f = bf16x4_to_float4(v[s]);
          mo.x += gs * f.x;
          mo.y += gs * f.y;
          mo.z += gs * f.z;
          mo.w += gs * f.w;
        }
    }
    hv = mo;
    h[(size_t)t * d4 + c] = hv;
    ss = hv.x * hv.x + hv.y * hv.y + hv.z * hv.z + hv.w * hv.w;
  }
  const float4 gg = ok ? ((const float4 *)gain)[c] : zero;  // in flight during the sum of squares
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const int nw = (blockDim.x + 31) >> 5;
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
  for (int w = 0; w < nw; ++w) tot += red[w];
  const float inv = rsqrtf(tot / (4 * d4) + eps);
  if (ok) {  // the next layer's QKV operand, in operand tiles
    __nv_bfloat162 p0 = __floats2bfloat162_rn(hv.x * inv * gg.x, hv.y * inv * gg.y);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(hv.z * inv * gg.z, hv.w * inv * gg.w);
    *(uint2 *)(x_tiles + tiled_index(T, 4 * d4, t, 4 * c)) = make_uint2(*(uint32_t *)&p0, *(uint32_t *)&p1);
  }
}


// 16-byte copies of [L][n][Hkv][hd] rows into the paged pools.
__global__ void kv_append_kernel(const uint4 *k_new, const uint4 *v_new, uint4 *k_pool,
                                 uint4 *v_pool, const int *page_table, int L, int n_pages, int pos0,
                                 int n, int Hkv, int hd, int pg) {
  pdl_wait();
  pdl_trigger();
  const int vec = hd / 8;  // uint4 per head row
  const size_t total = (size_t)L * n * Hkv * vec;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % vec);
    size_t r = i / vec;
    const int h = (int)(r % Hkv);
    r /= Hkv;
    const int t = (int)(r % n);
    const int l = (int)(r / n);
    const int p = pos0 + t, s = p % pg;
    // (page, head) block: hd/64 sub-blocks [pg][64], 16-byte chunk c of slot
    // s at chunk position c ^ (s % 8)
    const size_t dst = (((size_t)l * n_pages + page_table[p / pg]) * Hkv + h) * pg * vec +
                       (size_t)(c >> 3) * pg * 8 + (size_t)s * 8 + ((c & 7) ^ (s & 7));
    k_pool[dst] = k_new[i];
    v_pool[dst] = v_new[i];
  }
}

}  // namespace

namespace {
thread_local bool t_pdl_suspended = false;
}

bool pdl_enabled() {
  static int on = -1;
  if (on < 0) {
    const char *v = getenv("DG_PDL");
    on = (v && v[0] == '1') ? 1 : 0;
  }
  return on == 1 && !t_pdl_suspended;
}

void pdl_suspend(bool suspended) { t_pdl_suspended = suspended; }

static float weight_scale(float std_dev) {
  return (float)((double)std_dev * sqrt(3.0) / 8388608.0);
}

cudaError_t fill_weights(bf16 *dst, uint64_t n, uint64_t seed, uint32_t tid, uint64_t e0,
                         float std_dev, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  fill_weights_kernel<<<grid_for(n, 256), 256, 0, st>>>(dst, n, (uint32_t)seed,
                                                        (uint32_t)(seed >> 32), tid, e0,
                                                        weight_scale(std_dev));
  return cudaGetLastError();
}

cudaError_t fill_tiled_weights(bf16 *dst, int rows, int cols, int r1, int r2, uint32_t tid0, uint32_t tid1,
                               uint32_t tid2, uint64_t seed, float std_dev, cudaStream_t st) {
  const uint64_t n = (uint64_t)rows * cols;
  if (n == 0) return cudaSuccess;
  if (cols % 64) return cudaErrorInvalidValue;
  fill_tiled_kernel<<<grid_for(n, 256), 256, 0, st>>>(dst, rows, cols, r1, r2, tid0, tid1, tid2, (uint32_t)seed,
                                                      (uint32_t)(seed >> 32), weight_scale(std_dev));
  return cudaGetLastError();
}

cudaError_t fill_moe_weights(bf16 *wr, bf16 *wgu, bf16 *wd, int d, int E, int F, int layer,
                             uint64_t seed, float std_dev, cudaStream_t st) {
  const uint32_t base = 100u + 16u * (uint32_t)layer;
  cudaError_t e = fill_tiled_weights(wr, E, d, E, E, base + 4, base + 4, base + 4, seed, std_dev, st);
  if (e != cudaSuccess) return e;
  const uint64_t n = (uint64_t)E * 2 * F * d;
  fill_gate_up_kernel<<<grid_for(n, 256), 256, 0, st>>>(wgu, E, F, d, (uint32_t)seed,
                                                        (uint32_t)(seed >> 32), base + 5, base + 6,
                                                        weight_scale(std_dev));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  fill_down_kernel<<<grid_for(n, 256), 256, 0, st>>>(wd, E, F, d, (uint32_t)seed, (uint32_t)(seed >> 32), base + 7,
                                                     weight_scale(std_dev));
  return cudaGetLastError();
}

cudaError_t fill_const(float *dst, size_t n, float v, cudaStream_t st) {
  fill_const_kernel<<<grid_for(n, 256), 256, 0, st>>>(dst, n, v);
  return cudaGetLastError();
}

cudaError_t rope_table(float *ct, float *stt, int max_pos, int hd, float base, cudaStream_t st) {
  const size_t n = (size_t)max_pos * (hd / 2);
  rope_table_kernel<<<grid_for(n, 256), 256, 0, st>>>(ct, stt, max_pos, hd / 2, hd, (double)base);
  return cudaGetLastError();
}

cudaError_t canvas_init(int *x, uint8_t *committed, int *last, int *stable, int C, int V,
                        uint64_t seed, int canvas, cudaStream_t st, int n_req) {
  return launch_pdl(canvas_init_kernel, dim3(ceil_div(C, 256), n_req), dim3(256), 0, st, x, committed, last, stable,
                    C, V, seed, canvas);
}

cudaError_t embed_rows(float *h, const bf16 *table, const int *ids, int T, int d, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(embed_kernel, dim3(T), dim3(256), 0, st, h, table, ids, d);
}

cudaError_t rmsnorm_rows(bf16 *out, const float *h, const float *gain, int T, int d, float eps,
                         cudaStream_t st, bf16 *out_lo, bool tiled) {
  if (T == 0) return cudaSuccess;
  if (d % 4 || (tiled && d % 64)) return cudaErrorInvalidValue;
  return launch_pdl(rmsnorm_kernel, dim3(T), dim3(kNormThreads), 0, st, out, out_lo, h, gain, d, eps,
                    tiled ? T : 0);
}


size_t moe_max_work(int T, int k, int E, int tile_rows) {
  return (size_t)(T * k + tile_rows - 1) / tile_rows + E;
}

size_t moe_work_ints(int T, int k, int E, int tile_rows) {
  return 3 * moe_max_work(T, k, E, tile_rows) + 1 + kFfnSplitUnits;
}


cudaError_t moe_combine(float *h, const bf16 *y, const float *gates, const int *slot_row, int T,
                        int k, int d, bool accumulate, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (k > 16 || d % 4) return cudaErrorInvalidValue;
  return launch_pdl(combine_kernel, dim3(T), dim3(256), 0, st, (float4 *)h, (const uint2 *)y, gates, slot_row, k,
                    d / 4, accumulate ? 1 : 0);
}

cudaError_t moe_combine_norm(float *h, const bf16 *y, const float *gates, const int *slot_row,
                             int T, int k, int d, const float *gain, float eps, bf16 *x_tiles,
                             cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (k > 16 || d % 64 || d > 4 * 1024) return cudaErrorInvalidValue;
  return launch_pdl(combine_norm_kernel, dim3(T), dim3((d / 4 + 31) & ~31), 0, st, (float4 *)h, (const uint2 *)y,
                    gates, slot_row, k, d / 4, gain, eps, x_tiles, T);
}


cudaError_t kv_append(const bf16 *k_new, const bf16 *v_new, bf16 *k_pool, bf16 *v_pool,
                      const int *page_table, int L, int n_pages, int pos0, int n, int Hkv, int hd,
                      int pg, cudaStream_t st) {
  const size_t total = (size_t)L * n * Hkv * (hd / 8);
  if (total == 0) return cudaSuccess;
  return launch_pdl(kv_append_kernel, dim3(grid_for(total, 256, 152 * 16)), dim3(256), 0, st,
                    (const uint4 *)k_new, (const uint4 *)v_new, (uint4 *)k_pool, (uint4 *)v_pool, page_table, L,
                    n_pages, pos0, n, Hkv, hd, pg);
}

}  // namespace dg
