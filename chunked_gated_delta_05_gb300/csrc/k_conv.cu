// Causal depthwise convolution + SiLU over the token axis (the short convolution that
// produces q, k and v ahead of the delta rule; hyper-parallel GDN Diff Coverage page,
// `_causal_conv1d_with_cp_halo` and the packed ShortConv path): for channel c of a row at
// position t of its sequence,
//   z[t][c] = bias[c] + sum_{i<W} w[c][i] x[t - (W-1-i) d][c],   y = z sigmoid(z) (SiLU),
// where positions before the sequence start read the sequence's halo (the (W-1) d tokens
// preceding it, e.g. the previous context-parallel rank's tail) or zero; packed documents
// never read across their boundaries.
//
// GB300 mapping: a memory-bound stencil. Rows are token-major [R][C] bf16, so a warp reads
// and writes whole 16-byte vectors of consecutive channels; each thread owns 8 channels of
// 64 consecutive rows and keeps the taps in registers, re-reading the W-1 preceding rows
// from L1. The backward materialises dz = dy silu'(z) in fp32, then forms dx from it, and
// the weight/bias gradients as per-tile partial sums reduced in a fixed order.
#include "common.cuh"
#include "conv.cuh"

namespace gdn {

namespace {

constexpr int kRowsPerTile = 64;
constexpr int kThreads = 64;   // x 8 channels = 512 channels per CTA column

// Sequence of row r: index n with cu[n] <= r < cu[n+1] (dense: r / T).
__device__ __forceinline__ int seq_of(const ConvParams& p, long long r) {
  if (!p.cu) return int(r / p.T);
  int lo = 0, hi = p.N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cu[mid] <= r) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}
__device__ __forceinline__ long long seq_start(const ConvParams& p, int n) {
  return p.cu ? (long long)p.cu[n] : (long long)n * p.T;
}
__device__ __forceinline__ long long seq_end(const ConvParams& p, int n) {
  return p.cu ? (long long)p.cu[n + 1] : (long long)(n + 1) * p.T;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* src, float* f) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(src));
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 t = __bfloat1622float2(b[e]);
    f[2 * e] = t.x;
    f[2 * e + 1] = t.y;
  }
}
__device__ __forceinline__ void store8(__nv_bfloat16* dst, const float* f) {
  uint4 u;
  __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) b[e] = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
  *reinterpret_cast<uint4*>(dst) = u;
}

// Input at sequence position `pos` (may be negative: the halo, or zero) for channels c..c+7.
__device__ __forceinline__ void input8(const ConvParams& p, int n, long long start, long long pos, int c,
                                       float* f) {
  if (pos >= 0) {
    load8(p.x + (start + pos) * p.C + c, f);
  } else if (p.halo && pos >= -p.HW) {
    load8(p.halo + ((long long)n * p.HW + (p.HW + pos)) * p.C + c, f);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = 0.f;
  }
}

// Pre-activation z of row r (sequence n starting at `start`) for channels c..c+7.
__device__ __forceinline__ void preact8(const ConvParams& p, int n, long long start, long long r, int c,
                                        const float (&w)[kConvMaxTaps][8], float* z) {
#pragma unroll
  for (int e = 0; e < 8; ++e) z[e] = p.bias ? p.bias[c + e] : 0.f;
  const long long pos = r - start;
#pragma unroll
  for (int i = 0; i < kConvMaxTaps; ++i) {
    if (i >= p.W) break;
    float x[8];
    input8(p, n, start, pos - (long long)(p.W - 1 - i) * p.dil, c, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) z[e] = fmaf(w[i][e], x[e], z[e]);
  }
}

__device__ __forceinline__ void load_taps(const ConvParams& p, int c, float (&w)[kConvMaxTaps][8]) {
#pragma unroll
  for (int i = 0; i < kConvMaxTaps; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) w[i][e] = i < p.W ? p.w[(c + e) * p.W + i] : 0.f;
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.f / (1.f + __expf(-z)); }

}  // namespace

__global__ void __launch_bounds__(kThreads) k_conv_fwd(const ConvParams p) {
  const int c = 8 * (blockIdx.y * kThreads + threadIdx.x);
  if (c >= p.C) return;
  float w[kConvMaxTaps][8];
  load_taps(p, c, w);
  const long long r0 = (long long)blockIdx.x * kRowsPerTile;
  const long long r1 = r0 + kRowsPerTile < p.R ? r0 + kRowsPerTile : p.R;
  int n = seq_of(p, r0);
  long long start = seq_start(p, n), end = seq_end(p, n);
  for (long long r = r0; r < r1; ++r) {
    while (r >= end) {  // next packed document
      ++n;
      start = end;
      end = seq_end(p, n);
    }
    float z[8];
    preact8(p, n, start, r, c, w, z);
    if (p.silu)
#pragma unroll
      for (int e = 0; e < 8; ++e) z[e] *= sigmoidf_(z[e]);
    store8(p.y + r * p.C + c, z);
  }
}

// Backward pass 1: dz = dy * silu'(z) (fp32, kept for pass 2) and the tile's partial sums of
// dbias = sum dz and dw[i] = sum dz x[t - (W-1-i) d].
__global__ void __launch_bounds__(kThreads) k_conv_dz(const ConvParams p) {
  const int c = 8 * (blockIdx.y * kThreads + threadIdx.x);
  if (c >= p.C) return;
  float w[kConvMaxTaps][8];
  load_taps(p, c, w);
  float gw[kConvMaxTaps][8], gb[8];
#pragma unroll
  for (int i = 0; i < kConvMaxTaps; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) gw[i][e] = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) gb[e] = 0.f;
  const long long r0 = (long long)blockIdx.x * kRowsPerTile;
  const long long r1 = r0 + kRowsPerTile < p.R ? r0 + kRowsPerTile : p.R;
  int n = seq_of(p, r0);
  long long start = seq_start(p, n), end = seq_end(p, n);
  for (long long r = r0; r < r1; ++r) {
    while (r >= end) {
      ++n;
      start = end;
      end = seq_end(p, n);
    }
    float z[8], dy[8];
    preact8(p, n, start, r, c, w, z);
    load8(p.dy + r * p.C + c, dy);
    float dz[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (p.silu) {
        const float s = sigmoidf_(z[e]);
        dz[e] = dy[e] * s * (1.f + z[e] * (1.f - s));
      } else {
        dz[e] = dy[e];
      }
      gb[e] += dz[e];
    }
    float4* o = reinterpret_cast<float4*>(p.dz + r * p.C + c);
    o[0] = make_float4(dz[0], dz[1], dz[2], dz[3]);
    o[1] = make_float4(dz[4], dz[5], dz[6], dz[7]);
    const long long pos = r - start;
#pragma unroll
    for (int i = 0; i < kConvMaxTaps; ++i) {
      if (i >= p.W) break;
      float x[8];
      input8(p, n, start, pos - (long long)(p.W - 1 - i) * p.dil, c, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) gw[i][e] = fmaf(dz[e], x[e], gw[i][e]);
    }
  }
  // partials [tile][C][W + 1]: the W tap sums then the bias sum
  float* part = p.part + (size_t(blockIdx.x) * p.C + c) * (p.W + 1);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
#pragma unroll
    for (int i = 0; i < kConvMaxTaps; ++i)
      if (i < p.W) part[e * (p.W + 1) + i] = gw[i][e];
    part[e * (p.W + 1) + p.W] = gb[e];
  }
}

// Backward pass 2: dx[s] = sum_i w[i] dz[s + (W-1-i) d] over outputs of the same sequence;
// rows at the start of a sequence also feed the halo gradient (next kernel).
__global__ void __launch_bounds__(kThreads) k_conv_dx(const ConvParams p) {
  const int c = 8 * (blockIdx.y * kThreads + threadIdx.x);
  if (c >= p.C) return;
  float w[kConvMaxTaps][8];
  load_taps(p, c, w);
  const long long r0 = (long long)blockIdx.x * kRowsPerTile;
  const long long r1 = r0 + kRowsPerTile < p.R ? r0 + kRowsPerTile : p.R;
  int n = seq_of(p, r0);
  long long start = seq_start(p, n), end = seq_end(p, n);
  for (long long s = r0; s < r1; ++s) {
    while (s >= end) {
      ++n;
      start = end;
      end = seq_end(p, n);
    }
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
    for (int i = 0; i < kConvMaxTaps; ++i) {
      if (i >= p.W) break;
      const long long t = s + (long long)(p.W - 1 - i) * p.dil;
      if (t < end) {
        const float4* d4 = reinterpret_cast<const float4*>(p.dz + t * p.C + c);
        const float4 a = __ldg(d4), b = __ldg(d4 + 1);
        const float dz[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(w[i][e], dz[e], acc[e]);
      }
    }
    store8(p.dx + s * p.C + c, acc);
  }
}

// Halo gradient: halo slot j of sequence n is position j - HW; it feeds outputs
// t = j - HW + (W-1-i) d in [0, len).
__global__ void __launch_bounds__(kThreads) k_conv_dhalo(const ConvParams p) {
  const int c = 8 * (blockIdx.y * kThreads + threadIdx.x);
  if (c >= p.C) return;
  const int n = blockIdx.x / p.HW, j = blockIdx.x % p.HW;
  float w[kConvMaxTaps][8];
  load_taps(p, c, w);
  const long long start = seq_start(p, n), len = seq_end(p, n) - start;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
  for (int i = 0; i < kConvMaxTaps; ++i) {
    if (i >= p.W) break;
    const long long t = (long long)j - p.HW + (long long)(p.W - 1 - i) * p.dil;
    if (t >= 0 && t < len) {
      const float* d = p.dz + (start + t) * p.C + c;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(w[i][e], d[e], acc[e]);
    }
  }
  float* o = p.dhalo + ((long long)n * p.HW + j) * p.C + c;
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = acc[e];
}

// dw, dbias: the tiles' partial sums, added in tile order (deterministic).
__global__ void __launch_bounds__(256) k_conv_reduce(const ConvParams p, int tiles) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;  // (c, i) with i = W for the bias
  if (idx >= p.C * (p.W + 1)) return;
  float acc = 0.f;
  for (int t = 0; t < tiles; ++t) acc += p.part[size_t(t) * p.C * (p.W + 1) + idx];
  const int c = idx / (p.W + 1), i = idx % (p.W + 1);
  if (i < p.W) p.dw[c * p.W + i] = acc;
  else if (p.dbias) p.dbias[c] = acc;
}

cudaError_t launch_conv_fwd(const ConvParams& p, cudaStream_t s) {
  dim3 grid(unsigned((p.R + kRowsPerTile - 1) / kRowsPerTile), unsigned((p.C / 8 + kThreads - 1) / kThreads));
  k_conv_fwd<<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_conv_bwd(const ConvParams& p, cudaStream_t s) {
  const unsigned tiles = unsigned((p.R + kRowsPerTile - 1) / kRowsPerTile);
  dim3 grid(tiles, unsigned((p.C / 8 + kThreads - 1) / kThreads));
  k_conv_dz<<<grid, kThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_conv_dx<<<grid, kThreads, 0, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.dhalo && p.HW > 0) {
    dim3 g2(unsigned(p.N * p.HW), grid.y);
    k_conv_dhalo<<<g2, kThreads, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  k_conv_reduce<<<(p.C * (p.W + 1) + 255) / 256, 256, 0, s>>>(p, int(tiles));
  return cudaGetLastError();
}

size_t conv_partials_bytes(long long R, int C, int W) {
  return size_t((R + kRowsPerTile - 1) / kRowsPerTile) * C * (W + 1) * 4;
}

}  // namespace gdn
