// Warp-level building blocks: the epilogue tile context of the tensor-core
// GEMMs and the cp.async / mma.sync helpers of the canvas attention kernel.
#pragma once
#include "common.cuh"

namespace dg {

// Context handed to the epilogue.
struct TileCtx {
  int m0, n0;      // tile origin in (M, N) of this group
  int m_valid;     // rows of the tile inside M
  int n_valid;     // columns of the tile inside the group's N
  int group;       // expert (0 if not grouped)
  int b_base;      // first B row of the group
  int swz;         // tile layout: element (f, t) at f * ldc + (t ^ (f & swz)); 0 or 31
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

}  // namespace dg
