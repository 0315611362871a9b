// Block-level vocabulary-tile partials used both by the LM-head GEMM epilogue
// (logits straight from the accumulators, never written to HBM) and by the
// standalone kernel that reduces given fp32 logits.
#pragma once
#include "common.cuh"

namespace dg {

// Per-row scratch needed next to the logits tile.
struct PartialScratch {
  float *kap;   // [R][ldl] Gumbel keys
  float *rm;    // [R] tile max
  int *ra;      // [R] first argmax
};

// L: shared fp32 [R][ldl] logits of one 256-wide vocab tile starting at v0;
// row r is canvas position pos0 + r and is stored at planes row (out_row0 + r).
// Overwrites L with dg_exp(l - m).  All threads of the block must call it.
__device__ __forceinline__ void block_tile_partials(float *L, int ldl, PartialScratch sc, int R,
                                                    int v0, int tile, int tiles, int pos0,
                                                    uint32_t ctr2, uint32_t key0, uint32_t key1,
                                                    const PartialPlanes &P, int out_row0) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  // 1. max and first argmax per row (order-free: value desc, index asc)
  for (int r = warp; r < R; r += nw) {
    float m = L[r * ldl + lane];
    int a = lane;
#pragma unroll
    for (int j = 1; j < kVocabTile / 32; ++j) {
      const float l = L[r * ldl + lane + 32 * j];
      if (l > m) {
        m = l;
        a = lane + 32 * j;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float mo = __shfl_xor_sync(0xffffffffu, m, off);
      const int ao = __shfl_xor_sync(0xffffffffu, a, off);
      if (mo > m || (mo == m && ao < a)) {
        m = mo;
        a = ao;
      }
    }
    if (lane == 0) {
      sc.rm[r] = m;
      sc.ra[r] = a;
    }
  }
  __syncthreads();
  // 2. elementwise: exponentials and Gumbel keys (one Philox call per 4 entries)
  for (int idx = tid; idx < R * (kVocabTile / 4); idx += nt) {
    const int r = idx / (kVocabTile / 4), q = idx % (kVocabTile / 4);
    const U4 w = philox10((uint32_t)(v0 / 4 + q), (uint32_t)(pos0 + r), ctr2, kTagGumbel, key0, key1);
    const float m = sc.rm[r];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int v = 4 * q + j;
      const float l = L[r * ldl + v];
      sc.kap[r * ldl + v] = fadd(l, gumbel(open_uniform(w.w[j])));
      L[r * ldl + v] = dg_exp(fsub(l, m));
    }
  }
  __syncthreads();
  // 3. sequential ascending sums (one thread per row) and Gumbel argmax
  for (int r = tid; r < 2 * R; r += nt) {
    if (r < R) {
      float s = 0.0f;
      for (int v = 0; v < kVocabTile; ++v) s = fadd(s, L[r * ldl + v]);
      const size_t o = (size_t)(out_row0 + r) * tiles + tile;
      P.m[o] = sc.rm[r];
      P.a[o] = v0 + sc.ra[r];
      P.s[o] = s;
    } else {
      const int rr = r - R;
      float gk = sc.kap[rr * ldl];
      int gi = 0;
      for (int v = 1; v < kVocabTile; ++v) {
        const float k = sc.kap[rr * ldl + v];
        if (k > gk) {
          gk = k;
          gi = v;
        }
      }
      const size_t o = (size_t)(out_row0 + rr) * tiles + tile;
      P.gk[o] = gk;
      P.gi[o] = v0 + gi;
    }
  }
}

}  // namespace dg
