// Token positions of the ring's blocks under the three layouts, for the
// fp32 kernels ("Ring Attention: the math", section "Causal masking, load
// balance, and other wrinkles"; "Ring attention, explained", section "The
// causal-mask catch").  A slice of N tokens is cut into P blocks of c = N / P
// rows; local row r of block j sits at token position
//   contiguous  j c + r
//   zigzag      chunk j (r < c/2) or chunk 2P - 1 - j of 2P chunks of c/2
//   striped     j + P r
// Under every layout the positions of a block increase along its rows.
#pragma once

#include <cstdint>

#include "ra_internal.h"

namespace ra {

// Position of local row r of block j.
__device__ __forceinline__ int64_t layout_pos(int layout, int64_t j, int64_t r, int64_t P,
                                              int64_t c) {
  if (layout == kZigzag) {
    const int64_t h = c / 2;
    return r < h ? j * h + r : (2 * P - 1 - j) * h + (r - h);
  }
  if (layout == kStriped) return j + P * r;
  return j * c + r;
}

// Block holding position n.
__device__ __forceinline__ int64_t layout_block(int layout, int64_t n, int64_t P, int64_t c) {
  if (layout == kZigzag) {
    const int64_t chunk = n / (c / 2);
    return chunk < P ? chunk : 2 * P - 1 - chunk;
  }
  if (layout == kStriped) return n % P;
  return n / c;
}

// Local row of position n inside its block.
__device__ __forceinline__ int64_t layout_local(int layout, int64_t n, int64_t P, int64_t c) {
  if (layout == kZigzag) {
    const int64_t h = c / 2;
    return (n / h < P ? 0 : h) + n % h;
  }
  if (layout == kStriped) return n / P;
  return n % c;
}

}  // namespace ra
