// Causal depthwise convolution + SiLU over the token axis (the short convolution that
// produces q, k and v ahead of the delta rule; hyper-parallel GDN Diff Coverage page,
// `_causal_conv1d_with_cp_halo` and the packed ShortConv path): for channel c of a row at
// position t of its sequence,
//   z[t][c] = bias[c] + sum_{i<W} w[c][i] x[t - (W-1-i) d][c],   y = z sigmoid(z) (SiLU),
// where positions before the sequence start read the sequence's halo (the (W-1) d tokens
// preceding it, e.g. the previous context-parallel rank's tail) or zero; packed documents
// never read across their boundaries.
//
// GB300 mapping: a memory-bound stencil. Rows are token-major [R][C] bf16 and a CTA covers 64
// rows of a 256-channel block, staged in shared memory with asynchronous 16-byte copies.
// - Unit dilation and up to 4 taps (the short convolution of the path): each warp walks a run
//   of 32 consecutive rows for 64 channels with register windows of the last W rows, so every
//   input is read from shared memory once; runs inside one sequence take a path with no
//   per-row checks. The backward is one pass: dz = dy silu'(z) stays in registers and dx of a
//   row is formed as soon as the dz it needs exist (k_conv_fwd_runs, k_conv_bwd_fused).
// - Other dilations and widths: the 8 warps of a CTA interleave its rows (16 bytes of a row
//   per lane), each thread keeps its 8 channels' taps in registers, and the backward
//   materialises dz in fp32, then forms dx from it.
// The weight/bias gradients are per-tile sums (over warps in shared memory, over tiles in a
// fixed order).
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

// ---------------------------------------------------------------- fused backward, unit dilation
// For d = 1 and W <= 4 the backward runs in one pass: the CTA stages x rows [r0 - HW, r0 + 64 + HW)
// and dy rows [r0, r0 + 64 + HW) of its 256-channel block (HW = W - 1), then each warp walks a
// run of 32 rows for 64 channels (2 per lane) with register windows of the last W inputs and
// the last W dz values: dz of row u comes from z (window) and dy, and as soon as dz of row
// t + HW exists, dx of row t = sum_k w'_k dz[t + k] (w'_k = w[W-1-k], the tap at offset k) is
// complete and stored. dz never leaves registers (rows of a sequence's first HW positions are
// written to the workspace for the halo gradient). The dz of a run's last HW rows is recomputed
// by the next run. Weight and bias sums per warp are added over the CTA's two runs in a fixed
// order and written as the tile's partials.
constexpr int kFuseRun = 32;                        // rows per warp
constexpr int kFuseRuns = kRowsPerTile / kFuseRun;  // 2 runs x 4 channel quarters = 8 warps

__device__ __forceinline__ float2 smem2(const uint8_t* tile, int row, int cl) {
  const uint32_t u = *reinterpret_cast<const uint32_t*>(tile + size_t(row) * (kBlockChannels * 2) + cl * 2);
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
}

// Input at sequence position pos < 0 for channels c, c+1: the sequence's halo or zero.
__device__ __forceinline__ float2 before_start2(const ConvParams& p, int n, long long pos, int c) {
  if (p.halo && pos >= -p.HW) {
    const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(p.halo + ((long long)n * p.HW + (p.HW + pos)) * p.C + c));
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
  }
  return make_float2(0.f, 0.f);
}

template <int W>
__global__ void __launch_bounds__(kThreads, 3) k_conv_bwd_fused(const ConvParams p) {
  extern __shared__ __align__(16) uint8_t s_tile[];
  constexpr int HW = W - 1;
  constexpr int kRowBytes = kBlockChannels * 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int quarter = warp & 3, run = warp >> 2;
  const int cb = blockIdx.x * kBlockChannels, cl = 64 * quarter + 2 * lane, c = cb + cl;
  const long long r0 = (long long)blockIdx.y * kRowsPerTile;
  uint8_t* s_x = s_tile;                                         // tile row i = global row r0 - HW + i
  uint8_t* s_dy = s_tile + (kRowsPerTile + 2 * HW) * kRowBytes;  // tile row i = global row r0 + i
  stage_rows<2>(p.x, p.R, p.C, cb, r0 - HW, kRowsPerTile + 2 * HW, s_x);
  stage_rows<2>(p.dy, p.R, p.C, cb, r0, kRowsPerTile + HW, s_dy);
  const bool active = c < p.C;
  // taps by offset: wk[k] multiplies the input k rows back
  float2 wk[W], bias = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < W; ++k)
    wk[k] = active ? make_float2(__ldg(p.w + c * W + (W - 1 - k)), __ldg(p.w + (c + 1) * W + (W - 1 - k)))
                   : make_float2(0.f, 0.f);
  if (active && p.bias) bias = make_float2(__ldg(p.bias + c), __ldg(p.bias + c + 1));
  float2 gw[W], gb = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < W; ++k) gw[k] = make_float2(0.f, 0.f);
  stage_wait();
  __syncthreads();
  const long long t0 = r0 + kFuseRun * run;
  if (active && t0 < p.R) {
    float2 xw[W], dzw[W];   // xw[k]: input of row u - k; dzw[j]: dz of row u - j
#pragma unroll
    for (int k = 0; k < W; ++k) {
      xw[k] = make_float2(0.f, 0.f);
      dzw[k] = make_float2(0.f, 0.f);
    }
    SeqCursor su(p, t0), st(p, t0);
    const long long pos0 = t0 - su.start;
    if (su.end >= t0 + kFuseRun + HW && !(p.dhalo && pos0 < HW)) {
      // Clean run: rows t0 .. t0 + kFuseRun + HW - 1 all lie in the sequence of t0, so no row
      // needs a cursor, a mask or a range check. The windows are circular (row t0 + s in slot
      // s % W), so the W-fold unrolled steps rename registers instead of moving them.
#pragma unroll
      for (int k = 1; k < W; ++k)
        xw[W - k] = pos0 >= k ? smem2(s_x, int(t0 - k - (r0 - HW)), cl) : before_start2(p, su.n, pos0 - k, c);
      const uint8_t* xs = s_x + size_t(t0 - (r0 - HW)) * kRowBytes;
      const uint8_t* ds = s_dy + size_t(t0 - r0) * kRowBytes;
      __nv_bfloat16* dxr = p.dx + t0 * p.C + c;
#pragma unroll 1
      for (int s0 = 0; s0 < kFuseRun + HW; s0 += W) {
#pragma unroll
        for (int j = 0; j < W; ++j) {
          const int s = s0 + j;
          if (s < kFuseRun + HW) {
            xw[j] = smem2(xs, s, cl);
            const float2 dy = smem2(ds, s, cl);
            float z0 = bias.x, z1 = bias.y;
#pragma unroll
            for (int k = 0; k < W; ++k) {
              z0 = fmaf(wk[k].x, xw[(j - k + W) % W].x, z0);
              z1 = fmaf(wk[k].y, xw[(j - k + W) % W].y, z1);
            }
            float2 dz = dy;
            if (p.silu) {
              const float s0g = sigmoidf_(z0), s1g = sigmoidf_(z1);
              dz.x = dy.x * s0g * (1.f + z0 * (1.f - s0g));
              dz.y = dy.y * s1g * (1.f + z1 * (1.f - s1g));
            }
            if (s < kFuseRun) {
              gb.x += dz.x;
              gb.y += dz.y;
#pragma unroll
              for (int k = 0; k < W; ++k) {
                gw[k].x = fmaf(dz.x, xw[(j - k + W) % W].x, gw[k].x);
                gw[k].y = fmaf(dz.y, xw[(j - k + W) % W].y, gw[k].y);
              }
            }
            dzw[j] = dz;
            if (s >= HW) {   // dx of row t0 + s - HW from dz of rows t0 + s - HW .. t0 + s
              float a0 = 0.f, a1 = 0.f;
#pragma unroll
              for (int k = 0; k < W; ++k) {
                a0 = fmaf(wk[k].x, dzw[(j - HW + k + W) % W].x, a0);
                a1 = fmaf(wk[k].y, dzw[(j - HW + k + W) % W].y, a1);
              }
              *reinterpret_cast<__nv_bfloat162*>(dxr) = __floats2bfloat162_rn(a0, a1);
              dxr += p.C;
            }
          }
        }
      }
    } else {
    {
      // the window as it stands before the first step's shift: xw[k - 1] = input at offset k
      // of row t0 (rows before its sequence's start read that sequence's halo or zero)
#pragma unroll
      for (int k = 1; k < W; ++k)
        xw[k - 1] = pos0 >= k ? smem2(s_x, int(t0 - k - (r0 - HW)), cl) : before_start2(p, su.n, pos0 - k, c);
    }
#pragma unroll 2
    for (int s = 0; s < kFuseRun + HW; ++s) {
      const long long u = t0 + s;
#pragma unroll
      for (int k = W - 1; k > 0; --k) {
        xw[k] = xw[k - 1];
        dzw[k] = dzw[k - 1];
      }
      float2 dz = make_float2(0.f, 0.f);
      if (u < p.R) {
        xw[0] = smem2(s_x, int(u - (r0 - HW)), cl);
        su.advance(p, u);
        const long long pos = u - su.start;
        if (pos == 0 && s > 0) {
          // a sequence starts at this row: the window's older entries become its halo or zero
#pragma unroll
          for (int k = 1; k < W; ++k) xw[k] = before_start2(p, su.n, -k, c);
        }
        const float2 dy = smem2(s_dy, int(u - r0), cl);
        float z0 = bias.x, z1 = bias.y;
#pragma unroll
        for (int k = 0; k < W; ++k) {
          z0 = fmaf(wk[k].x, xw[k].x, z0);
          z1 = fmaf(wk[k].y, xw[k].y, z1);
        }
        if (p.silu) {
          const float s0 = sigmoidf_(z0), s1 = sigmoidf_(z1);
          dz.x = dy.x * s0 * (1.f + z0 * (1.f - s0));
          dz.y = dy.y * s1 * (1.f + z1 * (1.f - s1));
        } else {
          dz = dy;
        }
        if (s < kFuseRun) {
          gb.x += dz.x;
          gb.y += dz.y;
#pragma unroll
          for (int k = 0; k < W; ++k) {
            gw[k].x = fmaf(dz.x, xw[k].x, gw[k].x);
            gw[k].y = fmaf(dz.y, xw[k].y, gw[k].y);
          }
          if (p.dhalo && pos < HW) *reinterpret_cast<float2*>(p.dz + u * p.C + c) = dz;
        }
      }
      dzw[0] = dz;
      const long long t = u - HW;   // dx of row t needs dz of rows t .. t + HW: complete now
      if (t >= t0 && t < p.R) {
        st.advance(p, t);
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int k = 0; k < W; ++k)
          if (t + k < st.end) {
            a0 = fmaf(wk[k].x, dzw[HW - k].x, a0);
            a1 = fmaf(wk[k].y, dzw[HW - k].y, a1);
          }
        *reinterpret_cast<__nv_bfloat162*>(p.dx + t * p.C + c) = __floats2bfloat162_rn(a0, a1);
      }
    }
    }
  }
  // partials of the tile: the two runs' sums per (channel, tap / bias), added in run order
  __syncthreads();   // the staged tiles are no longer read: reuse them for the exchange
  float* s_part = reinterpret_cast<float*>(s_tile);   // [run][256 channels][W + 1]
  {
    float* d0 = s_part + (size_t(run) * kBlockChannels + cl) * (W + 1);
    float* d1 = d0 + (W + 1);
#pragma unroll
    for (int k = 0; k < W; ++k) {   // tap index i = W - 1 - k
      d0[W - 1 - k] = gw[k].x;
      d1[W - 1 - k] = gw[k].y;
    }
    d0[W] = gb.x;
    d1[W] = gb.y;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < kBlockChannels * (W + 1); idx += kThreads) {
    const int ch = idx / (W + 1), slot = idx % (W + 1);
    if (cb + ch >= p.C) continue;
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < kFuseRuns; ++q) acc += s_part[(size_t(q) * kBlockChannels + ch) * (W + 1) + slot];
    p.part[(size_t(blockIdx.y) * p.C + cb + ch) * (W + 1) + slot] = acc;
  }
}

// Forward for unit dilation and W <= 4, in the same layout: the CTA stages x rows
// [r0 - HW, r0 + 64) of its 256-channel block, each warp walks a run of 32 rows for 64
// channels (2 per lane) with a register window of the last W inputs. A run inside one sequence
// takes the clean path (circular window, no per-row checks); a run that meets a sequence start
// or the last row shifts its window and patches it with the new sequence's halo or zero.
template <int W>
__global__ void __launch_bounds__(kThreads) k_conv_fwd_runs(const ConvParams p) {
  extern __shared__ __align__(16) uint8_t s_tile[];   // tile row i = global row r0 - HW + i
  constexpr int HW = W - 1;
  constexpr int kRowBytes = kBlockChannels * 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int quarter = warp & 3, run = warp >> 2;
  const int cb = blockIdx.x * kBlockChannels, cl = 64 * quarter + 2 * lane, c = cb + cl;
  const long long r0 = (long long)blockIdx.y * kRowsPerTile;
  stage_rows<2>(p.x, p.R, p.C, cb, r0 - HW, kRowsPerTile + HW, s_tile);
  const bool active = c < p.C;
  float2 wk[W], bias = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < W; ++k)
    wk[k] = active ? make_float2(__ldg(p.w + c * W + (W - 1 - k)), __ldg(p.w + (c + 1) * W + (W - 1 - k)))
                   : make_float2(0.f, 0.f);
  if (active && p.bias) bias = make_float2(__ldg(p.bias + c), __ldg(p.bias + c + 1));
  stage_wait();
  __syncthreads();
  const long long t0 = r0 + kFuseRun * run;
  if (!active || t0 >= p.R) return;   // no barrier follows
  float2 xw[W];
#pragma unroll
  for (int k = 0; k < W; ++k) xw[k] = make_float2(0.f, 0.f);
  SeqCursor su(p, t0);
  const long long pos0 = t0 - su.start;
  if (su.end >= t0 + kFuseRun) {
#pragma unroll
    for (int k = 1; k < W; ++k)
      xw[W - k] = pos0 >= k ? smem2(s_tile, int(t0 - k - (r0 - HW)), cl) : before_start2(p, su.n, pos0 - k, c);
    const uint8_t* xs = s_tile + size_t(t0 - (r0 - HW)) * kRowBytes;
    __nv_bfloat16* yr = p.y + t0 * p.C + c;
#pragma unroll 1
    for (int s0 = 0; s0 < kFuseRun; s0 += W) {
#pragma unroll
      for (int j = 0; j < W; ++j) {
        const int s = s0 + j;
        if (s < kFuseRun) {
          xw[j] = smem2(xs, s, cl);
          float z0 = bias.x, z1 = bias.y;
#pragma unroll
          for (int k = 0; k < W; ++k) {
            z0 = fmaf(wk[k].x, xw[(j - k + W) % W].x, z0);
            z1 = fmaf(wk[k].y, xw[(j - k + W) % W].y, z1);
          }
          if (p.silu) {
            z0 = __fdividef(z0, 1.f + __expf(-z0));
            z1 = __fdividef(z1, 1.f + __expf(-z1));
          }
          *reinterpret_cast<__nv_bfloat162*>(yr) = __floats2bfloat162_rn(z0, z1);
          yr += p.C;
        }
      }
    }
    return;
  }
#pragma unroll
  for (int k = 1; k < W; ++k)
    xw[k - 1] = pos0 >= k ? smem2(s_tile, int(t0 - k - (r0 - HW)), cl) : before_start2(p, su.n, pos0 - k, c);
#pragma unroll 1
  for (int s = 0; s < kFuseRun; ++s) {
    const long long u = t0 + s;
    if (u >= p.R) break;
#pragma unroll
    for (int k = W - 1; k > 0; --k) xw[k] = xw[k - 1];
    xw[0] = smem2(s_tile, int(u - (r0 - HW)), cl);
    su.advance(p, u);
    if (u == su.start && s > 0) {
      // a sequence starts at this row: the window's older entries become its halo or zero
#pragma unroll
      for (int k = 1; k < W; ++k) xw[k] = before_start2(p, su.n, -k, c);
    }
    float z0 = bias.x, z1 = bias.y;
#pragma unroll
    for (int k = 0; k < W; ++k) {
      z0 = fmaf(wk[k].x, xw[k].x, z0);
      z1 = fmaf(wk[k].y, xw[k].y, z1);
    }
    if (p.silu) {
      z0 = __fdividef(z0, 1.f + __expf(-z0));
      z1 = __fdividef(z1, 1.f + __expf(-z1));
    }
    *reinterpret_cast<__nv_bfloat162*>(p.y + u * p.C + c) = __floats2bfloat162_rn(z0, z1);
  }
}

template <int W>
cudaError_t conv_fwd_runs(const ConvParams& p, cudaStream_t s) {
  dim3 grid(unsigned((p.C + kBlockChannels - 1) / kBlockChannels), unsigned((p.R + kRowsPerTile - 1) / kRowsPerTile));
  const size_t smem = size_t(kRowsPerTile + W - 1) * kBlockChannels * 2;
  k_conv_fwd_runs<W><<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int W>
cudaError_t conv_bwd_fused(const ConvParams& p, cudaStream_t s) {
  const unsigned tiles = unsigned((p.R + kRowsPerTile - 1) / kRowsPerTile);
  dim3 grid(unsigned((p.C + kBlockChannels - 1) / kBlockChannels), tiles);
  const size_t smem = size_t(2 * kRowsPerTile + 3 * (W - 1)) * kBlockChannels * 2;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_conv_bwd_fused<W>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  k_conv_bwd_fused<W><<<grid, kThreads, smem, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.dhalo && p.HW > 0) {
    dim3 g2(grid.x, unsigned((p.N * p.HW + kWarps - 1) / kWarps));
    k_conv_dhalo<4><<<g2, kThreads, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  k_conv_reduce<<<(p.C * (p.W + 1) + 255) / 256, 256, 0, s>>>(p, int(tiles));
  return cudaGetLastError();
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
  if (p.dil == 1) {
    switch (p.W) {
      case 1: return conv_fwd_runs<1>(p, s);
      case 2: return conv_fwd_runs<2>(p, s);
      case 3: return conv_fwd_runs<3>(p, s);
      case 4: return conv_fwd_runs<4>(p, s);
      default: break;
    }
  }
  return p.W <= 4 ? conv_fwd_mw<4>(p, s) : conv_fwd_mw<kConvMaxTaps>(p, s);
}

cudaError_t launch_conv_bwd(const ConvParams& p, cudaStream_t s) {
  if (p.dil == 1) {
    switch (p.W) {
      case 1: return conv_bwd_fused<1>(p, s);
      case 2: return conv_bwd_fused<2>(p, s);
      case 3: return conv_bwd_fused<3>(p, s);
      case 4: return conv_bwd_fused<4>(p, s);
      default: break;
    }
  }
  return p.W <= 4 ? conv_bwd_mw<4>(p, s) : conv_bwd_mw<kConvMaxTaps>(p, s);
}

size_t conv_partials_bytes(long long R, int C, int W) {
  return size_t((R + kRowsPerTile - 1) / kRowsPerTile) * C * (W + 1) * 4;
}

}  // namespace gdn
