// Causal depthwise convolution + SiLU over the token axis (the short convolution that
// produces q, k and v ahead of the delta rule; hyper-parallel GDN Diff Coverage page,
// `_causal_conv1d_with_cp_halo` and the packed ShortConv path): for channel c of a row at
// position t of its sequence,
//   z[t][c] = bias[c] + sum_{i<W} w[c][i] x[t - (W-1-i) d][c],   y = z sigmoid(z) (SiLU),
// where positions before the sequence start read the sequence's halo (the (W-1) d tokens
// preceding it, e.g. the previous context-parallel rank's tail) or zero; packed documents
// never read across their boundaries.
//
// GB300 mapping: a memory-bound stencil with every output row independent. Rows are
// token-major [R][C] bf16; a warp takes whole rows of a 256-channel block (16 bytes per lane),
// the 8 warps of a CTA interleave 64 consecutive rows so the W-row input windows overlap in
// L1, and each thread keeps its 8 channels' taps in registers. The backward materialises
// dz = dy silu'(z) in fp32, then forms dx from it, and the weight/bias gradients as per-tile
// sums (over warps in shared memory, over tiles in a fixed order).
#include "common.cuh"
#include "conv.cuh"

namespace gdn {

namespace {

// A CTA covers 64 rows x 256 channels: warp w takes rows w, w + 8, ..., lane l channels
// 8 l .. 8 l + 7 of the CTA's block, so a warp reads and writes 512 contiguous bytes per row and
// the 8 warps read overlapping row windows from L1.
constexpr int kRowsPerTile = 64;
constexpr int kWarps = 8;
constexpr int kBlockChannels = 256;
constexpr int kThreads = 32 * kWarps;

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
template <int MW>
__device__ __forceinline__ void preact8(const ConvParams& p, int n, long long start, long long r, int c,
                                        const float (&w)[MW][8], float* z) {
#pragma unroll
  for (int e = 0; e < 8; ++e) z[e] = p.bias ? __ldg(p.bias + c + e) : 0.f;
  const long long pos = r - start;
#pragma unroll
  for (int i = 0; i < MW; ++i) {
    if (i >= p.W) break;
    float x[8];
    input8(p, n, start, pos - (long long)(p.W - 1 - i) * p.dil, c, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) z[e] = fmaf(w[i][e], x[e], z[e]);
  }
}

template <int MW>
__device__ __forceinline__ void load_taps(const ConvParams& p, int c, float (&w)[MW][8]) {
#pragma unroll
  for (int i = 0; i < MW; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) w[i][e] = i < p.W ? __ldg(p.w + (c + e) * p.W + i) : 0.f;
}

// sigmoid(z) = 1 / (1 + e^-z) with the fast reciprocal division (-> 0 for z -> -inf, 1 for +inf)
__device__ __forceinline__ float sigmoidf_(float z) { return __fdividef(1.f, 1.f + __expf(-z)); }

// Sequence bookkeeping of one thread walking increasing rows (a packed document changes rarely).
struct SeqCursor {
  int n;
  long long start, end;
  __device__ __forceinline__ SeqCursor(const ConvParams& p, long long r) {
    n = seq_of(p, r);
    start = seq_start(p, n);
    end = seq_end(p, n);
  }
  __device__ __forceinline__ void advance(const ConvParams& p, long long r) {
    while (r >= end) {
      ++n;
      start = end;
      end = seq_end(p, n);
    }
  }
};

}  // namespace

template <int MW>
__global__ void __launch_bounds__(kThreads) k_conv_fwd(const ConvParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x * kBlockChannels + 8 * lane;
  if (c >= p.C) return;
  float w[MW][8];
  load_taps(p, c, w);
  const long long r0 = (long long)blockIdx.y * kRowsPerTile;
#pragma unroll 2
  for (int j = 0; j < kRowsPerTile / kWarps; ++j) {
    const long long r = r0 + warp + kWarps * j;
    if (r >= p.R) break;
    const int n = seq_of(p, r);
    float z[8];
    preact8(p, n, seq_start(p, n), r, c, w, z);
    if (p.silu)
#pragma unroll
      for (int e = 0; e < 8; ++e) z[e] *= sigmoidf_(z[e]);
    store8(p.y + r * p.C + c, z);
  }
}

// Backward pass 1: dz = dy * silu'(z) (fp32, kept for pass 2) and the tile's sums of
// dbias = sum dz and dw[i] = sum dz x[t - (W-1-i) d], reduced over the warps in shared memory.
template <int MW>
__global__ void __launch_bounds__(kThreads) k_conv_dz(const ConvParams p) {
  constexpr int kSlots = 5;   // (tap or bias) sums exchanged per shared-memory pass
  __shared__ float s_part[kWarps][32][kSlots * 8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x * kBlockChannels + 8 * lane;
  const bool active = c < p.C;
  float gw[MW][8], gb[8];
#pragma unroll
  for (int i = 0; i < MW; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) gw[i][e] = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) gb[e] = 0.f;
  if (active) {
    float w[MW][8];
    load_taps(p, c, w);
    const long long r0 = (long long)blockIdx.y * kRowsPerTile;
#pragma unroll 2
    for (int j = 0; j < kRowsPerTile / kWarps; ++j) {
      const long long r = r0 + warp + kWarps * j;
      if (r >= p.R) break;
      const int n = seq_of(p, r);
      const long long start = seq_start(p, n);
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
      for (int i = 0; i < MW; ++i) {
        if (i >= p.W) break;
        float x[8];
        input8(p, n, start, pos - (long long)(p.W - 1 - i) * p.dil, c, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) gw[i][e] = fmaf(dz[e], x[e], gw[i][e]);
      }
    }
  }
  // partials [tile][C][W + 1] (the W tap sums, then the bias sum), summed over the warps in
  // warp order through shared memory, kSlots slots of 8 channels per pass
  for (int s0 = 0; s0 <= MW; s0 += kSlots) {
#pragma unroll
    for (int q = 0; q < kSlots; ++q) {
      const int slot = s0 + q;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float v = 0.f;
#pragma unroll
        for (int i = 0; i < MW; ++i)
          if (slot == i) v = gw[i][e];
        if (slot == MW) v = gb[e];
        s_part[warp][lane][q * 8 + e] = v;
      }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < 32 * 8 * kSlots; idx += kThreads) {
      const int q = idx % kSlots, cl = idx / kSlots;   // slot in this pass, channel in the block
      const int slot = s0 + q;
      const int cc = blockIdx.x * kBlockChannels + cl;
      // slot MW is the bias; slots p.W .. MW-1 are taps this problem does not have
      const int out = slot == MW ? p.W : slot;
      if (cc >= p.C || slot > MW || (slot < MW && slot >= p.W)) continue;
      float acc = 0.f;
      for (int wq = 0; wq < kWarps; ++wq) acc += s_part[wq][cl >> 3][q * 8 + (cl & 7)];
      p.part[(size_t(blockIdx.y) * p.C + cc) * (p.W + 1) + out] = acc;
    }
    __syncthreads();
  }
}

// Backward pass 2: dx[s] = sum_i w[i] dz[s + (W-1-i) d] over outputs of the same sequence.
template <int MW>
__global__ void __launch_bounds__(kThreads) k_conv_dx(const ConvParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x * kBlockChannels + 8 * lane;
  if (c >= p.C) return;
  float w[MW][8];
  load_taps(p, c, w);
  const long long r0 = (long long)blockIdx.y * kRowsPerTile;
#pragma unroll 2
  for (int j = 0; j < kRowsPerTile / kWarps; ++j) {
    const long long s = r0 + warp + kWarps * j;
    if (s >= p.R) break;
    const long long end = seq_end(p, seq_of(p, s));
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
    for (int i = 0; i < MW; ++i) {
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
template <int MW>
__global__ void __launch_bounds__(kThreads) k_conv_dhalo(const ConvParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x * kBlockChannels + 8 * lane;
  const int row = blockIdx.y * kWarps + warp;   // (n, j) flattened
  if (c >= p.C || row >= p.N * p.HW) return;
  const int n = row / p.HW, j = row % p.HW;
  float w[MW][8];
  load_taps(p, c, w);
  const long long start = seq_start(p, n), len = seq_end(p, n) - start;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
  for (int i = 0; i < MW; ++i) {
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

// ---------------------------------------------------------------- shared-memory tiled path
// (halo HW = (W-1) d <= 64 rows): the CTA stages rows [r0 - HW, r0 + 64) of its 256-channel
// block once with coalesced 16-byte loads, then every output row reads its taps from there;
// taps before a sequence's start read the halo or zero instead.
constexpr int kMaxTileHalo = 64;

// Stages rows [row0, row0 + nrows) of a 256-channel block of a [R][C] tensor with `es`-byte
// elements into `tile` ([nrows][256 * es] bytes) with asynchronous 16-byte copies, all in flight
// at once (rows outside [0, R) and channels past C are zero-filled); the caller waits with
// stage_wait() and a barrier.
template <int es>
__device__ __forceinline__ void stage_rows(const void* src, long long R, int C, int cb, long long row0, int nrows,
                                           uint8_t* tile) {
  constexpr int vec_per_row = kBlockChannels * es / 16;
  const int nvec = nrows * vec_per_row;
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(tile));
  for (int idx = threadIdx.x; idx < nvec; idx += kThreads) {
    const int rr = idx / vec_per_row, v = idx % vec_per_row;
    const long long row = row0 + rr;
    const int ch = cb + v * (16 / es);
    const bool ok = row >= 0 && row < R && ch < C;
    const char* g = static_cast<const char*>(src) + (ok ? (row * C + ch) * es : 0);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(base + idx * 16), "l"(g), "r"(ok ? 16 : 0)
                 : "memory");
  }
}
__device__ __forceinline__ void stage_wait() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The block's taps: channels cb .. cb+255 are one contiguous [256][W] fp32 range of the [C][W]
// weights, i.e. 8 W floats per lane. They are staged with 16-byte copies into rows of 8 W + 4
// floats per lane (the 16-byte pad puts eight consecutive lanes' float4 reads on distinct
// banks), then each thread reads its own row.
template <int MW>
__device__ __forceinline__ void stage_taps(const ConvParams& p, int cb, float* s_w) {
  const int nch = min(kBlockChannels, p.C - cb);
  const int per_lane = 2 * p.W;                    // float4 chunks of a lane's 8 W floats
  const int nvec = (nch / 8) * per_lane;
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(s_w));
  const char* g = reinterpret_cast<const char*>(p.w + size_t(cb) * p.W);
  for (int idx = threadIdx.x; idx < nvec; idx += kThreads) {
    const int ln = idx / per_lane, k = idx % per_lane;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(base + (ln * (8 * MW + 4) + 4 * k) * 4),
                 "l"(g + idx * 16)
                 : "memory");
  }
}
// This thread's 8 channels x MW taps from the staged block, and its 8 biases.
template <int MW>
__device__ __forceinline__ void taps_from(const ConvParams& p, const float* s_w, int lane, float (&w)[MW][8],
                                          float* bias) {
  float row[8 * MW];
  const float4* r4 = reinterpret_cast<const float4*>(s_w + lane * (8 * MW + 4));
#pragma unroll
  for (int k = 0; k < 2 * MW; ++k) {
    const float4 v = r4[k];
    row[4 * k] = v.x; row[4 * k + 1] = v.y; row[4 * k + 2] = v.z; row[4 * k + 3] = v.w;
  }
  // the staged row holds channel e's taps at e * W + i
#pragma unroll
  for (int i = 0; i < MW; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float t = 0.f;
#pragma unroll
      for (int ww = 1; ww <= MW; ++ww)
        if (ww == p.W && i < ww) t = row[e * ww + i];
      w[i][e] = t;
    }
  if (bias) {
    if (p.bias) {
      const int c = blockIdx.x * kBlockChannels + 8 * lane;
      const float4 b0 = __ldg(reinterpret_cast<const float4*>(p.bias + c));
      const float4 b1 = __ldg(reinterpret_cast<const float4*>(p.bias + c) + 1);
      bias[0] = b0.x; bias[1] = b0.y; bias[2] = b0.z; bias[3] = b0.w;
      bias[4] = b1.x; bias[5] = b1.y; bias[6] = b1.z; bias[7] = b1.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) bias[e] = 0.f;
    }
  }
}


__device__ __forceinline__ void smem8(const uint8_t* tile, int row, int lane, float* f) {
  const uint4 u = reinterpret_cast<const uint4*>(tile)[row * 32 + lane];
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 t = __bfloat1622float2(b[e]);
    f[2 * e] = t.x;
    f[2 * e + 1] = t.y;
  }
}

// z of row r from the staged tile (tile row 0 = global row r0 - HW).
template <int MW>
__device__ __forceinline__ void preact8_tiled(const ConvParams& p, const uint8_t* tile, long long r0, int n,
                                              long long start, long long r, int c, int lane,
                                              const float (&w)[MW][8], const float* bias, float* z) {
#pragma unroll
  for (int e = 0; e < 8; ++e) z[e] = bias[e];
  const long long pos = r - start;
#pragma unroll
  for (int i = 0; i < MW; ++i) {
    if (i >= p.W) break;
    const long long sp = pos - (long long)(p.W - 1 - i) * p.dil;
    float x[8];
    if (sp >= 0) smem8(tile, int(r - (long long)(p.W - 1 - i) * p.dil - (r0 - p.HW)), lane, x);
    else input8(p, n, start, sp, c, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) z[e] = fmaf(w[i][e], x[e], z[e]);
  }
}

template <int MW>
__global__ void __launch_bounds__(kThreads, 3) k_conv_fwd_tiled(const ConvParams p) {
  extern __shared__ __align__(16) uint8_t s_tile[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cb = blockIdx.x * kBlockChannels, c = cb + 8 * lane;
  const long long r0 = (long long)blockIdx.y * kRowsPerTile;
  __shared__ __align__(16) float s_w[32 * (8 * MW + 4)];
  stage_rows<2>(p.x, p.R, p.C, cb, r0 - p.HW, kRowsPerTile + p.HW, s_tile);
  stage_taps<MW>(p, cb, s_w);
  stage_wait();
  __syncthreads();
  if (c >= p.C) return;
  float w[MW][8], bias[8];
  taps_from(p, s_w, lane, w, bias);
  SeqCursor sq(p, r0 + warp < p.R ? r0 + warp : p.R - 1);
#pragma unroll 2
  for (int j = 0; j < kRowsPerTile / kWarps; ++j) {
    const long long r = r0 + warp + kWarps * j;
    if (r >= p.R) break;
    sq.advance(p, r);
    float z[8];
    preact8_tiled(p, s_tile, r0, sq.n, sq.start, r, c, lane, w, bias, z);
    if (p.silu)
#pragma unroll
      for (int e = 0; e < 8; ++e) z[e] = __fdividef(z[e], 1.f + __expf(-z[e]));
    store8(p.y + r * p.C + c, z);
  }
}

template <int MW>
__global__ void __launch_bounds__(kThreads, 2) k_conv_dz_tiled(const ConvParams p) {
  extern __shared__ __align__(16) uint8_t s_tile[];
  constexpr int kSlots = 5;
  __shared__ float s_part[kWarps][32][kSlots * 8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cb = blockIdx.x * kBlockChannels, c = cb + 8 * lane;
  const long long r0 = (long long)blockIdx.y * kRowsPerTile;
  uint8_t* s_dy = s_tile + (kRowsPerTile + p.HW) * kBlockChannels * 2;
  __shared__ __align__(16) float s_w[32 * (8 * MW + 4)];
  stage_rows<2>(p.x, p.R, p.C, cb, r0 - p.HW, kRowsPerTile + p.HW, s_tile);
  stage_rows<2>(p.dy, p.R, p.C, cb, r0, kRowsPerTile, s_dy);
  stage_taps<MW>(p, cb, s_w);
  stage_wait();
  __syncthreads();
  const bool active = c < p.C;
  float gw[MW][8], gb[8];
#pragma unroll
  for (int i = 0; i < MW; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) gw[i][e] = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) gb[e] = 0.f;
  if (active) {
    float w[MW][8], bias[8];
    taps_from(p, s_w, lane, w, bias);
    SeqCursor sq(p, r0 + warp < p.R ? r0 + warp : p.R - 1);
#pragma unroll 2
    for (int j = 0; j < kRowsPerTile / kWarps; ++j) {
      const long long r = r0 + warp + kWarps * j;
      if (r >= p.R) break;
      sq.advance(p, r);
      const int n = sq.n;
      const long long start = sq.start;
      float z[8], dy[8];
      preact8_tiled(p, s_tile, r0, n, start, r, c, lane, w, bias, z);
      smem8(s_dy, int(r - r0), lane, dy);
      float dz[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (p.silu) {
          const float sg = sigmoidf_(z[e]);
          dz[e] = dy[e] * sg * (1.f + z[e] * (1.f - sg));
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
      for (int i = 0; i < MW; ++i) {
        if (i >= p.W) break;
        const long long sp = pos - (long long)(p.W - 1 - i) * p.dil;
        float x[8];
        if (sp >= 0) smem8(s_tile, int(r - (long long)(p.W - 1 - i) * p.dil - (r0 - p.HW)), lane, x);
        else input8(p, n, start, sp, c, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) gw[i][e] = fmaf(dz[e], x[e], gw[i][e]);
      }
    }
  }
  for (int s0 = 0; s0 <= MW; s0 += kSlots) {
#pragma unroll
    for (int q = 0; q < kSlots; ++q) {
      const int slot = s0 + q;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float v = 0.f;
#pragma unroll
        for (int i = 0; i < MW; ++i)
          if (slot == i) v = gw[i][e];
        if (slot == MW) v = gb[e];
        s_part[warp][lane][q * 8 + e] = v;
      }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < 32 * 8 * kSlots; idx += kThreads) {
      const int q = idx % kSlots, cl = idx / kSlots;
      const int slot = s0 + q;
      const int cc = cb + cl;
      const int out = slot == MW ? p.W : slot;
      if (cc >= p.C || slot > MW || (slot < MW && slot >= p.W)) continue;
      float acc = 0.f;
      for (int wq = 0; wq < kWarps; ++wq) acc += s_part[wq][cl >> 3][q * 8 + (cl & 7)];
      p.part[(size_t(blockIdx.y) * p.C + cc) * (p.W + 1) + out] = acc;
    }
    __syncthreads();
  }
}

template <int MW>
__global__ void __launch_bounds__(kThreads, 3) k_conv_dx_tiled(const ConvParams p) {
  extern __shared__ __align__(16) uint8_t s_tile[];   // dz rows [r0, r0 + 64 + HW), fp32
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cb = blockIdx.x * kBlockChannels, c = cb + 8 * lane;
  const long long r0 = (long long)blockIdx.y * kRowsPerTile;
  __shared__ __align__(16) float s_w[32 * (8 * MW + 4)];
  stage_rows<4>(p.dz, p.R, p.C, cb, r0, kRowsPerTile + p.HW, s_tile);
  stage_taps<MW>(p, cb, s_w);
  stage_wait();
  __syncthreads();
  if (c >= p.C) return;
  float w[MW][8];
  taps_from(p, s_w, lane, w, static_cast<float*>(nullptr));
  const float4* t4 = reinterpret_cast<const float4*>(s_tile);
  SeqCursor sq(p, r0 + warp < p.R ? r0 + warp : p.R - 1);
#pragma unroll 2
  for (int j = 0; j < kRowsPerTile / kWarps; ++j) {
    const long long s = r0 + warp + kWarps * j;
    if (s >= p.R) break;
    sq.advance(p, s);
    const long long end = sq.end;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
    for (int i = 0; i < MW; ++i) {
      if (i >= p.W) break;
      const long long t = s + (long long)(p.W - 1 - i) * p.dil;
      if (t < end) {
        const int tr = int(t - r0);
        const float4 a = t4[(tr * 32 + lane) * 2], b = t4[(tr * 32 + lane) * 2 + 1];
        const float dz[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(w[i][e], dz[e], acc[e]);
      }
    }
    store8(p.dx + s * p.C + c, acc);
  }
}

template <int MW>
cudaError_t conv_fwd_mw(const ConvParams& p, cudaStream_t s) {
  dim3 grid(unsigned((p.C + kBlockChannels - 1) / kBlockChannels), unsigned((p.R + kRowsPerTile - 1) / kRowsPerTile));
  if (p.HW <= kMaxTileHalo) {
    const size_t smem = size_t(kRowsPerTile + p.HW) * kBlockChannels * 2;
    static bool attr = false;
    if (!attr) {
      cudaError_t e = cudaFuncSetAttribute(k_conv_fwd_tiled<MW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (kRowsPerTile + kMaxTileHalo) * kBlockChannels * 2);
      if (e != cudaSuccess) return e;
      attr = true;
    }
    k_conv_fwd_tiled<MW><<<grid, kThreads, smem, s>>>(p);
  } else {
    k_conv_fwd<MW><<<grid, kThreads, 0, s>>>(p);
  }
  return cudaGetLastError();
}

template <int MW>
cudaError_t conv_bwd_mw(const ConvParams& p, cudaStream_t s) {
  const unsigned tiles = unsigned((p.R + kRowsPerTile - 1) / kRowsPerTile);
  dim3 grid(unsigned((p.C + kBlockChannels - 1) / kBlockChannels), tiles);
  cudaError_t e;
  if (p.HW <= kMaxTileHalo) {
    static bool attr = false;
    if (!attr) {
      e = cudaFuncSetAttribute(k_conv_dz_tiled<MW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (2 * kRowsPerTile + kMaxTileHalo) * kBlockChannels * 2);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(k_conv_dx_tiled<MW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (kRowsPerTile + kMaxTileHalo) * kBlockChannels * 4);
      if (e != cudaSuccess) return e;
      attr = true;
    }
    k_conv_dz_tiled<MW><<<grid, kThreads, size_t(2 * kRowsPerTile + p.HW) * kBlockChannels * 2, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k_conv_dx_tiled<MW><<<grid, kThreads, size_t(kRowsPerTile + p.HW) * kBlockChannels * 4, s>>>(p);
  } else {
    k_conv_dz<MW><<<grid, kThreads, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k_conv_dx<MW><<<grid, kThreads, 0, s>>>(p);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.dhalo && p.HW > 0) {
    dim3 g2(grid.x, unsigned((p.N * p.HW + kWarps - 1) / kWarps));
    k_conv_dhalo<MW><<<g2, kThreads, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  k_conv_reduce<<<(p.C * (p.W + 1) + 255) / 256, 256, 0, s>>>(p, int(tiles));
  return cudaGetLastError();
}

// Kernels compiled for up to 4 taps (registers for the common short convolution) or 8.
cudaError_t launch_conv_fwd(const ConvParams& p, cudaStream_t s) {
  return p.W <= 4 ? conv_fwd_mw<4>(p, s) : conv_fwd_mw<kConvMaxTaps>(p, s);
}

cudaError_t launch_conv_bwd(const ConvParams& p, cudaStream_t s) {
  return p.W <= 4 ? conv_bwd_mw<4>(p, s) : conv_bwd_mw<kConvMaxTaps>(p, s);
}

size_t conv_partials_bytes(long long R, int C, int W) {
  return size_t((R + kRowsPerTile - 1) / kRowsPerTile) * C * (W + 1) * 4;
}

}  // namespace gdn
