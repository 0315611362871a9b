// Device-side building blocks shared by the kernels of the GB300 decoder:
// bf16 helpers, the Philox4x32-10 generator, the sampler's fp32 exp/log and
// the merge of vocabulary-tile partials of the commit / re-noise sampler.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace dg {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): ten rounds of the Philox-4x32 S-box
//   (c0,c1,c2,c3) -> (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0))
// with the key advanced by the Weyl increments after each round.
// ---------------------------------------------------------------------------
struct U4 {
  uint32_t w[4];
};

__host__ __device__ __forceinline__ U4 philox10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    c1 = (uint32_t)p1;
    c3 = (uint32_t)p0;
    c0 = n0;
    c2 = n2;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  U4 r;
  r.w[0] = c0; r.w[1] = c1; r.w[2] = c2; r.w[3] = c3;
  return r;
}

// Stream tags of the counter's fourth word.
constexpr uint32_t kTagWeight = 1, kTagInit = 2, kTagGumbel = 3;

// ---------------------------------------------------------------------------
// Sampler arithmetic.  Every operation is an explicitly rounded IEEE fp32
// intrinsic so that no contraction or approximation can change the bits.
//
// dg_exp: Cody & Waite (1980) range reduction  k = floor(x log2 e + 1/2),
// r = (x - k C1) - k C2 with ln 2 = C1 + C2, C1 = 355/512 (9 bits, so k C1
// is exact); e^r by its degree-7 Taylor polynomial (coefficients 1/j!) in
// Horner form; times 2^k assembled from the exponent bits.  NaN passes,
// x < -87 gives 0, x > 88 gives +inf.
//
// dg_log: x = 2^e m with m in [sqrt(1/2), sqrt(2)]; log m = 2 atanh(s),
// s = (m-1)/(m+1), by the odd series s + s^3/3 + ... + s^11/11 (Horner in
// s^2); log x = (e C2 + log m) + e C1.
// ---------------------------------------------------------------------------
constexpr double kLn2d = 0.6931471805599453;
constexpr float kLog2e = (float)(1.0 / kLn2d);
constexpr float kLn2Hi = (float)(355.0 / 512.0);
constexpr float kLn2Lo = (float)(kLn2d - 355.0 / 512.0);
constexpr float kSqrt2 = (float)1.4142135623730951;

__device__ __forceinline__ float fadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float fsub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float fmul(float a, float b) { return __fmul_rn(a, b); }

// Both are written without branches: the special cases are selected after
// the main path, so a warp evaluating many entries keeps them interleaved.
// The results are those of the branching form bit for bit (checked over all
// 2^32 inputs).
__device__ __forceinline__ float dg_exp(float x) {
  const float xc = fminf(fmaxf(x, -87.0f), 88.0f);
  const float kf = floorf(fadd(fmul(xc, kLog2e), 0.5f));
  float r = fsub(xc, fmul(kf, kLn2Hi));
  r = fsub(r, fmul(kf, kLn2Lo));
  float p = (float)(1.0 / 5040.0);
  p = fadd(fmul(p, r), (float)(1.0 / 720.0));
  p = fadd(fmul(p, r), (float)(1.0 / 120.0));
  p = fadd(fmul(p, r), (float)(1.0 / 24.0));
  p = fadd(fmul(p, r), (float)(1.0 / 6.0));
  p = fadd(fmul(p, r), 0.5f);
  p = fadd(fmul(p, r), 1.0f);
  p = fadd(fmul(p, r), 1.0f);
  const int k = (int)kf;
  float y = fmul(p, __int_as_float((k + 127) << 23));
  y = x < -87.0f ? 0.0f : y;
  y = x > 88.0f ? __int_as_float(0x7f800000) : y;
  return x != x ? x : y;
}

__device__ __forceinline__ float dg_log(float x) {
  const bool sub = x < 1.17549435e-38f;  // subnormal: scale into the normal range
  const float xs = sub ? fmul(x, 8388608.0f) : x;
  const int bits = __float_as_int(xs);
  int e = ((bits >> 23) & 0xff) - 127 - (sub ? 23 : 0);
  float m = __int_as_float((bits & 0x7fffff) | 0x3f800000);
  const bool big = m > kSqrt2;
  m = big ? fmul(m, 0.5f) : m;
  e += big ? 1 : 0;
  const float s = __fdiv_rn(fsub(m, 1.0f), fadd(m, 1.0f));
  const float z = fmul(s, s);
  float q = (float)(1.0 / 11.0);
  q = fadd(fmul(q, z), (float)(1.0 / 9.0));
  q = fadd(fmul(q, z), (float)(1.0 / 7.0));
  q = fadd(fmul(q, z), (float)(1.0 / 5.0));
  q = fadd(fmul(q, z), (float)(1.0 / 3.0));
  q = fmul(q, z);
  float lm = fadd(s, fmul(s, q));
  lm = fadd(lm, lm);
  const float ef = (float)e;
  float r = fadd(fadd(fmul(ef, kLn2Lo), lm), fmul(ef, kLn2Hi));
  r = x == 0.0f ? __int_as_float(0xff800000) : r;
  r = x < 0.0f ? __int_as_float(0x7fc00000) : r;
  r = x == __int_as_float(0x7f800000) ? x : r;
  return x != x ? x : r;
}

// Open-interval uniform of a Philox word: (2 (w >> 9) + 1) * 2^-24.
__device__ __forceinline__ float open_uniform(uint32_t w) {
  return fmul((float)(((w >> 9) << 1) | 1u), 5.9604644775390625e-08f);
}

__device__ __forceinline__ float gumbel(float u) { return -dg_log(-dg_log(u)); }

// ---------------------------------------------------------------------------
// Vocabulary-tile partials (tiles of 256 entries) and their merge.
// m = max, a = first index at the max, s = left-to-right fp32 sum of
// dg_exp(l - m), (gk, gi) = max / first argmax of l + Gumbel noise.
// ---------------------------------------------------------------------------
constexpr int kVocabTile = 256;

struct Partial {
  float m;
  int a;
  float s;
  float gk;
  int gi;
};

__device__ __forceinline__ Partial empty_partial() {
  Partial p;
  p.m = __int_as_float(0xff800000);
  p.a = 0;
  p.s = 0.0f;
  p.gk = __int_as_float(0xff800000);
  p.gi = 0;
  return p;
}

// Counter word 2 of the Gumbel stream for step n (1-based) of canvas k.
__host__ __device__ __forceinline__ uint32_t gumbel_ctr2(int canvas, int step) {
  return ((uint32_t)canvas << 16) | (uint32_t)step;
}

// Per-step sampler parameters kept in device memory, so that a captured
// denoising step can be replayed for every step of a canvas: Gumbel counter
// word 2, Philox key of the sample seed, 1-based step number, and 1 / the
// re-noise temperature of that step.
struct StepParams {
  uint32_t ctr2, key0, key1;
  int step;
  float inv_tau;
};

// Merge of two adjacent ranges, L the lower vocab range.  An empty right
// operand (m = -inf) leaves L unchanged.
__device__ __forceinline__ Partial merge_partials(const Partial &L, const Partial &R) {
  if (!(R.m > __int_as_float(0xff800000))) return L;
  Partial o;
  const float M = fmaxf(L.m, R.m);
  o.m = M;
  o.s = fadd(fmul(L.s, dg_exp(fsub(L.m, M))), fmul(R.s, dg_exp(fsub(R.m, M))));
  o.a = (R.m > L.m) ? R.a : L.a;
  if (R.gk > L.gk) {
    o.gk = R.gk;
    o.gi = R.gi;
  } else {
    o.gk = L.gk;
    o.gi = L.gi;
  }
  return o;
}

// Partials planes: m, a, s, gk, gi, each [rows][tiles].
struct PartialPlanes {
  float *m;
  int *a;
  float *s;
  float *gk;
  int *gi;
  __host__ __device__ static PartialPlanes at(void *base, int rows, int tiles) {
    PartialPlanes P;
    const size_t n = (size_t)rows * tiles;
    P.m = (float *)base;
    P.a = (int *)(P.m + n);
    P.s = (float *)(P.a + n);
    P.gk = (float *)(P.s + n);
    P.gi = (int *)(P.gk + n);
    return P;
  }
  __device__ __forceinline__ Partial load(size_t idx) const {
    Partial p;
    p.m = m[idx];
    p.a = a[idx];
    p.s = s[idx];
    p.gk = gk[idx];
    p.gi = gi[idx];
    return p;
  }
};

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + __expf(-x)); }

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// Programmatic dependent launch, opt-in (DG_PDL=1).  With it, the kernels of
// a denoising step are launched with programmatic stream serialization
// (launch_pdl), so a kernel's blocks may be resident while its predecessor in
// the stream is still running.  It is off by default: with it on, steps over
// long prefixes (32k tokens) and multi-request steps stalled on the GB300
// (a bounded wait of the attention gave up, and some runs did not return)
// while the same launches without it ran to the end; the cause is not known.
// Every such kernel calls pdl_wait() before it reads or writes anything an
// earlier kernel touches (griddepcontrol.wait returns once the preceding grid
// has completed and its memory is visible; it is a no-op for an ordinary
// launch) and pdl_trigger() once its own successor may be scheduled.
// ---------------------------------------------------------------------------
// Codes >= kShapeErrorBase in a device error word mean that a kernel found
// itself launched without the cluster shape it was built for (it returned
// before any cluster operation); lower codes are bounded waits that gave up.
constexpr int kShapeErrorBase = 200;

// The device error word of bounded waits, loaded at a kernel's start so that
// its latency overlaps the setup (a kernel that finds it set skips its waits:
// an earlier one already gave up).  Under programmatic dependent launch the
// load may precede the previous kernel's last write; a missed record only
// costs bounded waits that give up again.
__device__ __forceinline__ int ld_err_word(const int *p) {
  int v = 0;
  if (p) asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// CTAs in this CTA's cluster (1 for a launch without clusters).
__device__ __forceinline__ uint32_t cluster_ctas() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(n));
  return n;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

bool pdl_enabled();  // host: on only when DG_PDL=1 is set in the environment and it is not suspended
void pdl_suspend(bool suspended);  // host: this thread's launches without programmatic dependence

// Operand tiles of a row-major [rows][cols] bf16 matrix (cols a multiple of
// 64), the layout every tensor-core operand of the decoder is stored in: row
// block b (128 rows; the last one rows % 128 when that is not 0) holds
// cols / 64 tiles of rows_b x 64 elements, contiguous per k-tile; inside a
// tile the 16-byte chunk c of row r sits at chunk position c ^ (r % 8) (the
// tensor core's 128-byte-swizzled shared-memory order), so one contiguous
// bulk copy stages a tile.  Element index of (r, c):
__host__ __device__ inline size_t tiled_index(int rows, int cols, int r, int c) {
  const int b = r >> 7, rr = r & 127, kt = c >> 6, cc = c & 63;
  const int rows_b = rows - 128 * b < 128 ? rows - 128 * b : 128;
  return (size_t)128 * cols * b + (size_t)rows_b * 64 * kt + (size_t)rr * 64 + (size_t)((((cc >> 3) ^ (rr & 7)) << 3) | (cc & 7));
}

// ---- e4m3 (FP8) expert path -------------------------------------------------
// A row (an output feature of W_gate / W_up, or a token row of the expert
// input) is stored as e4m3(row * 2^-k) with k the smallest integer such that
// max|row| <= 448 * 2^k; conversion rounds to nearest even and saturates.
// An e4m3 matrix [R][C] in operand tiles occupies the bytes of a bf16 matrix
// [R][C/2] in operand tiles: 128-row blocks of 128-byte rows (128 elements
// per k-tile), 16-element chunk j of row r at chunk position j ^ (r % 8).
__device__ __forceinline__ int e4m3_scale_exp(float absmax) {
  if (!(absmax > 0.0f)) return 0;
  int e;
  const float m = frexpf(absmax, &e);  // absmax = m 2^e, 448 * 2^(e-9) = 0.875 * 2^e
  return m <= 0.875f ? e - 9 : e - 8;
}

// Two e4m3 codes: `lo` in the low byte (the lower address), `hi` in the high.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Byte offset of e4m3 element (r, c), c a multiple of 16, in operand tiles of [rows][cols].
__host__ __device__ inline size_t tiled_index_e4m3(int rows, int cols, int r, int c) {
  return 2 * tiled_index(rows, cols / 2, r, c / 2);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace dg
