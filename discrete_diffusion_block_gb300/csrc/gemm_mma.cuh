// The epilogue tile context of the tensor-core GEMMs.
#pragma once
#include "common.cuh"

namespace dg {

// Context handed to the epilogue.
struct TileCtx {
  int m0, n0;      // tile origin in (M, N)
  int m_valid;     // rows of the tile inside M
  int n_valid;     // columns of the tile inside N
  int swz;         // tile layout: element (f, t) at f * ldc + (t ^ (f & swz)); 0 or 31
  int prepared;    // the epilogue's prepare() already staged its inputs in its scratch
};

}  // namespace dg
