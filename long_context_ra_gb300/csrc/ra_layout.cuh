// Token positions of the ring's blocks under the three layouts ("Ring Attention: the math", section "Causal masking, load
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

// Heaviest-first numbering of the causal work units of one slice.  A unit
// is tile t of block b (tiles per block), numbered r = b tiles + t in launch
// order; under the mask a query tile's work grows with its positions and a
// key tile's shrinks with them, so the units are remapped to descending
// positions (desc: query tiles) or ascending ones (key tiles), and the last
// units to start are the lightest.  Contiguous: blocks in order.  Zigzag
// (block b holds chunks b and 2P-1-b, tiles / 2 tiles each; tiles even):
// chunks in order.  Striped (positions P r + b): tiles in order, the blocks
// interleaved.  A bijection of [0, P) x [0, tiles).
__device__ __forceinline__ void causal_order(int layout, int P, int tiles, bool desc, int& b,
                                             int& t) {
  const int r = b * tiles + t;
  if (layout == kZigzag && tiles % 2 == 0) {
    const int tpc = tiles / 2;
    const int k = desc ? 2 * P - 1 - r / tpc : r / tpc;  // chunk
    const int q = desc ? tpc - 1 - r % tpc : r % tpc;    // tile within the chunk
    b = k < P ? k : 2 * P - 1 - k;
    t = (k < P ? 0 : tpc) + q;
  } else if (layout == kStriped) {
    t = desc ? tiles - 1 - r / P : r / P;
    b = desc ? P - 1 - r % P : r % P;
  } else if (desc) {
    b = P - 1 - b;
    t = tiles - 1 - t;
  }
}

}  // namespace ra
