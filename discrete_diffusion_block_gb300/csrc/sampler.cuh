// The per-(row, vocabulary tile) reduction of the sampler, written once and
// used both by the LM-head epilogue (logits read straight from the tensor
// memory accumulator, never written to HBM) and by the standalone kernel that
// reduces given fp32 logits, so that injected-logit tests run the decoder's
// own reduction code.
#pragma once
#include "common.cuh"

namespace dg {

// Upper bound of the Gumbel noise of every Philox word whose top byte is b:
// the noise of word w is G(w) = -dg_log(-dg_log(open_uniform(w))), and G is
// strictly increasing in w >> 9 over all 2^23 values (checked exhaustively on
// the host against the oracle's fp32 transform, and the device transform
// against the oracle's bit for bit), so its value at the largest word of the
// bucket bounds the whole bucket.  The Gumbel-max scan computes the exact key
// only where l + bound can beat the running maximum; as fp32 addition is
// monotone, l + G(w) <= l + bound, and the winner and its key are the same as
// with every key computed.
__device__ __forceinline__ float gumbel_bucket_bound(int b) {
  return gumbel(open_uniform(((uint32_t)b << 24) | 0x00FFFFFFu));
}

// Partials of one row of one 256-wide vocabulary tile (tile index v, vocab
// entries 256 v .. 256 v + 255, canvas position pos):
//   m = max logit, a = first index reaching it (ascending v),
//   s = left-to-right fp32 sum of dg_exp(l - m),
//   (gk, gi) = max and first argmax of fp32(l * inv_tau) + G with the Gumbel
//              noise of the Philox words at counter (v * 64 + j / 4, pos, c2,
//              tag) word j % 4 (inv_tau = 1: exactly l + G).
// The 256 logits are read through `src` in eight chunks of 32:
//   src.issue(c, x) starts loading logits 32 c .. 32 c + 31 into x (bit patterns),
//   src.wait(x)     completes that load.
// gbound: the 256 bucket bounds of gumbel_bucket_bound (shared memory).
// Pass 1 per chunk: the eight Philox calls first (independent chains the
// scheduler can interleave with the load), then a branch-free max scan, then
// exact keys only for the columns whose bound beats the running maximum --
// gk only grows along the scan, so the bound against its value at the chunk
// start selects a superset of the columns needed.  Pass 2 re-reads the
// logits for the ascending sum of dg_exp(l - m).
template <class Src>
__device__ __forceinline__ Partial row_tile_partial(Src &src, int v, uint32_t pos, uint32_t c2,
                                                    uint32_t k0, uint32_t k1, const float *gbound,
                                                    float inv_tau) {
  float m = 0.0f, gk = 0.0f;
  int a = 0, gi = 0;
  const uint32_t w0 = (uint32_t)v * (kVocabTile / 4);
#pragma unroll 1
  for (int c = 0; c < kVocabTile / 32; ++c) {
    uint32_t x[32], wd[32];
    src.issue(c, x);
#pragma unroll
    for (int j4 = 0; j4 < 8; ++j4) {
      const U4 w = philox10(w0 + (uint32_t)(8 * c + j4), pos, c2, kTagGumbel, k0, k1);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) wd[4 * j4 + jj] = w.w[jj];
    }
    src.wait(x);
    int j0 = 0;
    if (c == 0) {
      m = __uint_as_float(x[0]);
      gk = fadd(fmul(m, inv_tau), gumbel(open_uniform(wd[0])));
      j0 = 1;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float l = __uint_as_float(x[j]);
      const bool up = j >= j0 && l > m;
      m = up ? l : m;
      a = up ? 32 * c + j : a;
    }
    uint32_t cand = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      cand |= (j >= j0 && fadd(fmul(__uint_as_float(x[j]), inv_tau), gbound[wd[j] >> 24]) > gk) ? (1u << j) : 0u;
    while (cand) {
      const int j = __ffs(cand) - 1;
      cand &= cand - 1;
      uint32_t xj = 0, wj = 0;
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        xj = t == j ? x[t] : xj;
        wj = t == j ? wd[t] : wj;
      }
      const float key = fadd(fmul(__uint_as_float(xj), inv_tau), gumbel(open_uniform(wj)));
      if (key > gk) {
        gk = key;
        gi = 32 * c + j;
      }
    }
  }
  float s = 0.0f;
#pragma unroll 1
  for (int c = 0; c < kVocabTile / 32; ++c) {
    uint32_t x[32];
    src.issue(c, x);
    src.wait(x);
    float ex[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) ex[j] = dg_exp(fsub(__uint_as_float(x[j]), m));
#pragma unroll
    for (int j = 0; j < 32; ++j) s = fadd(s, ex[j]);
  }
  Partial p;
  p.m = m;
  p.a = v * kVocabTile + a;
  p.s = s;
  p.gk = gk;
  p.gi = v * kVocabTile + gi;
  return p;
}

}  // namespace dg
