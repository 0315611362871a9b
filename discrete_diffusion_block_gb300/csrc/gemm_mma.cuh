// The epilogue tile context of the tensor-core GEMMs.
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
  int prepared;    // the epilogue's prepare() already staged its inputs in its scratch
};

}  // namespace dg
