// Unit-lower-triangular inverse of a chunk's 64x64 L, one column per lane pair (shared by the
// scalar-gate and per-channel-gate prepare kernels).
#pragma once
#include "common.cuh"

namespace gdn {

// Column `c` of X = (I + L)^-1 for a 64x64 strictly lower L, written to column c of sX
// (row-major [64][64] fp32) by a lane pair: lanes l and l ^ 16 of a warp hold the same column
// (part 0 and 1) and split the products with the already solved rows by parity, so one warp
// covers 16 columns. LT is L transposed (LT[j][i] = L[i][j]) so that the 16 rows of a tile
// read one column of L as four broadcast float4 loads. Forward substitution by 16-row tiles:
// y = -L[tile, :16b] X[:16b, c] (the pair's partial sums meet through one shuffle), then both
// lanes solve the 16x16 diagonal block in registers (x_c = 1, x_r = 0 above the diagonal,
// x_r = y_r - sum_j L[r][j] x_j below it, applied row by row as each x_j is final) and each
// writes back eight of its rows.
__device__ __forceinline__ void unit_lower_inverse_column(const float* __restrict__ LT, float* sX, int c,
                                                          int part) {
  const int c0 = c & ~15;  // warp-uniform: X[j][c] = 0 for j < c is already in sX
  for (int b = 0; b < 4; ++b) {
    const int r0 = 16 * b;
    float x[16];
    if (r0 + 15 < c0) {  // above the diagonal for the whole warp
#pragma unroll
      for (int e = 0; e < 16; ++e) x[e] = 0.f;
    } else {
      float y[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) y[e] = 0.f;
      // r0 - c0 is a multiple of 16, so both lanes of a pair run the same trip count
#pragma unroll 2
      for (int j = c0 + part; j < r0; j += 2) {
        const float xj = sX[j * kC + c];
        const float4* l4 = reinterpret_cast<const float4*>(LT + j * kC + r0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 l = l4[q];
          y[4 * q] = fmaf(-l.x, xj, y[4 * q]);
          y[4 * q + 1] = fmaf(-l.y, xj, y[4 * q + 1]);
          y[4 * q + 2] = fmaf(-l.z, xj, y[4 * q + 2]);
          y[4 * q + 3] = fmaf(-l.w, xj, y[4 * q + 3]);
        }
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) y[e] += __shfl_xor_sync(0xffffffffu, y[e], 16);
      // the 16x16 diagonal block, right-looking: row j is final once the rows above it have
      // been applied, and it then updates the rows below it from one line of L^T (the 16-byte
      // chunks that hold those rows), so the dependent chain is one FMA per row
#pragma unroll
      for (int e = 0; e < 16; ++e) x[e] = y[e];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int R = r0 + j;
        x[j] = (R < c) ? 0.f : ((R == c) ? 1.f : x[j]);
        if (j < 15) {
          const float4* l4 = reinterpret_cast<const float4*>(LT + (r0 + j) * kC + r0);
          float l[16];
#pragma unroll
          for (int q = (j + 1) / 4; q < 4; ++q) {
            const float4 v = l4[q];
            l[4 * q] = v.x;
            l[4 * q + 1] = v.y;
            l[4 * q + 2] = v.z;
            l[4 * q + 3] = v.w;
          }
#pragma unroll
          for (int r = j + 1; r < 16; ++r) x[r] = fmaf(-l[r], x[j], x[r]);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) sX[(r0 + 8 * part + e) * kC + c] = part ? x[8 + e] : x[e];
    __syncwarp();
  }
}

}  // namespace gdn
