// Backward, feature-major part: per chunk, the products contracted over the value dimension
// that involve the carried state, computed with the key/value feature on the 128 TMEM lanes.
//
// With h the state entering the chunk (K x V), dh' the gradient w.r.t. the state leaving it,
// v_new / dv_new the chunk's corrected values and their gradient, dO the output gradient and
// A = (I + L)^-1, the chunk map's adjoint gives (see the forward chain kernel for the map):
//   dQt  = dO h^T            (gradient of the gated, scaled queries)
//   dW   = -dv_new h^T       (gradient of k_cumdecay = W)
//   dKt  = v_new dh'^T       (gradient of the end-decayed keys)
//   dK1  = A^T dW            (gradient of beta exp(G) k^, the right factor of W = A K1)
//   dV1  = A^T dv_new        (gradient of beta v,        the right factor of U = A V1)
//   dgam = sum over v of h (.) dh'   (per key row; summed over keys for the scalar gate)
// GB300 mapping: one CTA per chunk and head, 256 threads; threads f and f + 128 own feature f
// (= TMEM lane f) and split its columns in halves. h and dh' rows are loaded by their lane
// owners and stored to TMEM as A operands of kind::tf32 MMAs (the chains save both in bf16, so
// the widened values are exact tf32 operands); dO^T, v_new, dv_new and A^T are SW128 K-major B
// operands in shared memory (v_new, dv_new by TMA). h and dh' arrive by TMA too (128-row boxes
// of 64 bf16 columns, 128-byte swizzle: a thread's column half is one panel row), so each
// thread reads its row from shared memory without bank conflicts. Results leave as token-major fp32 rows [t][f] (coalesced: the 128
// threads of one token row write 512 contiguous bytes; dQt, dKt and dK1, which only the
// token-major backward's CUDA-core assembly reads, are bf16: 256 bytes per row, each store two
// adjacent columns).
// (An L2 prefetch of the next wave's inputs made the whole step slower: with the heads split
// over two streams it competes with the other group's kernels.)
#include "common.cuh"
#include "umma.cuh"

namespace gdn {

namespace {

constexpr int kThreads = 256;
// [dO ; dv_new] as one 128-row operand [t][v] tf32, 4 panels x 128 rows (64 KB): rows 0-63 dO
// (converted from the bf16 tile), rows 64-127 dv_new (TMA), so h dO^T and h dv_new^T are one
// N = 128 product.
constexpr uint32_t kOffC = 0;
constexpr uint32_t kOffVN = 65536;    // v_new [t][v] (TMA), 4 panels x 64 rows
constexpr uint32_t kOffAT = 98304;    // A^T  [j][i] tf32, 2 panels x 64 rows (16 KB)
constexpr uint32_t kOffDO16 = 114688; // dO   [t][v] bf16 (TMA), 2 panels x 64 rows (16 KB)
constexpr uint32_t kOffHS = 131072;   // h [f][v] bf16, 2 panels x 128 rows (32 KB)
constexpr uint32_t kOffDH = kOffHS + 32768;  // dh' [f][v] bf16, 2 panels x 128 rows (32 KB)
constexpr uint32_t kSmemBytes = kOffDH + 32768 + 1024;
constexpr uint32_t kTH = 0, kTDH = 128, kTP1 = 256, kTP2 = 320, kTP3 = 384, kTP5 = 448;
static_assert(kTP2 == kTP1 + 64, "h [dO ; dv_new]^T lands in P1 | P2");

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    k_bwd_feat(const __grid_constant__ CUtensorMap mVN, const __grid_constant__ CUtensorMap mDVN,
               const __grid_constant__ CUtensorMap mdO, const __grid_constant__ CUtensorMap mH,
               const __grid_constant__ CUtensorMap mDH, const BwdFeatParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1k(smem_raw);
  __shared__ uint64_t bar_tma, bar_tma2, bar_mma, bar_mma3;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;
  __shared__ float s_red[8];
  __shared__ float s_dg[kThreads];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // heads fastest: the CTAs in flight share token rows of dO and neighbouring tiles
  const int c = int(blockIdx.x / p.hgn), h = int(blockIdx.x % p.hgn) + p.hg0, H = p.H;
  const size_t tile = size_t(c) * H + h;
  const int f = tid & 127, hf = tid >> 7;  // feature (TMEM lane) and column half
  const ChunkEntry ch = chunk_entry(p.chunks, c, p.dense_T);  // requested first: the dO load below waits on it

  if (warp == 0) tmem_alloc(&tslot, 512);
  if (tid == 0) {
    // the barriers are this thread's alone until the block barrier below: start the loads now.
    // First group: h, dh', dv_new, dO; v_new (read by the third product only) on its own barrier.
    abort_flag = 0;
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_tma2, 1);
    mbar_init(&bar_mma, 1);
    mbar_init(&bar_mma3, 1);
    fence_mbar_init();
    mbar_expect_tx(&bar_tma, 2u * 32768u + 32768u + 16384u);
    const int yh = int(tile) * kD;
    for (int pp = 0; pp < 2; ++pp) {
      tma_load_2d(sm + kOffHS + pp * 16384, &mH, pp * 64, yh, &bar_tma);
      tma_load_2d(sm + kOffDH + pp * 16384, &mDH, pp * 64, yh, &bar_tma);
    }
    for (int pp = 0; pp < 4; ++pp) tma_load_2d(sm + kOffC + pp * 16384 + 8192, &mDVN, pp * 32, int(tile) * kC, &bar_tma);
    for (int pp = 0; pp < 2; ++pp) tma_load_2d(sm + kOffDO16 + pp * 8192, &mdO, h * kD + 64 * pp, ch.x, &bar_tma);
    mbar_expect_tx(&bar_tma2, 32768u);
    for (int pp = 0; pp < 4; ++pp) tma_load_2d(sm + kOffVN + pp * 8192, &mVN, pp * 32, int(tile) * kC, &bar_tma2);
    prefetch_l2(p.A + tile * kTileAqk, 4u * kTileAqk);  // read after the first products are issued
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  const uint32_t tl = tb + tmem_lane_base(warp);
  // Half hf of the h and dh' rows f (panel hf of each: shared memory -> TMEM as tf32 A
  // operands, widened exactly from bf16); dgam partial sums in fp32.
  const bool tma_ok = mbar_wait(&bar_tma, 0, &abort_flag, p.status, kDevTimeoutTma);
  float dg = 0.f;
  if (tma_ok) {
    const uint8_t* hrow = sm + kOffHS + hf * 16384;
    const uint8_t* drow = sm + kOffDH + hf * 16384;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float a[32], b[32];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = 32 * q + 8 * e;
        const uint4 x = *reinterpret_cast<const uint4*>(hrow + sw128_offset(f, col, 128, 2));
        const uint4 y = *reinterpret_cast<const uint4*>(drow + sw128_offset(f, col, 128, 2));
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          // two bf16 per word, the lower column in the low half
          const float x0 = __uint_as_float(xs[u] << 16), x1 = __uint_as_float(xs[u] & 0xffff0000u);
          const float y0 = __uint_as_float(ys[u] << 16), y1 = __uint_as_float(ys[u] & 0xffff0000u);
          dg = fmaf(x0, y0, dg);
          dg = fmaf(x1, y1, dg);
          a[8 * e + 2 * u] = x0;
          a[8 * e + 2 * u + 1] = x1;
          b[8 * e + 2 * u] = y0;
          b[8 * e + 2 * u + 1] = y1;
        }
      }
      tmem_st32(tl + kTH + 64 * hf + 32 * q, a);
      tmem_st32(tl + kTDH + 64 * hf + 32 * q, b);
    }
  }
  // dO^T operand: element (t, v=f) of the K-major [t][v] tile from the bf16 TMA tile (half hf
  // of the tokens); rows past the chunk (the next document's, or out of range) are zero.
  if (tma_ok) {
#pragma unroll 8
    for (int t = 32 * hf; t < 32 * hf + 32; ++t) {
      const float x = t < ch.y ? __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
                                     sm + kOffDO16 + sw128_offset(t, f, kC, 2)))
                               : 0.f;
      *reinterpret_cast<float*>(sm + kOffC + sw128_offset(t, f, 2 * kC, 4)) = x;
    }
  }
  tmem_wait_st();
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // [P1 | P2] (kTP2 = kTP1 + 64) = h [dO ; dv_new]^T from thread 0; P3 = dh' v_new^T from
  // thread 32 once v_new has landed, with its own barrier, so that everything up to the second
  // product group proceeds meanwhile
  if (tid == 0) {
    if (tma_ok) {
      tc_fence_after();
      const uint32_t id128 = idesc_tf32(128, 128), sC = smem_u32(sm + kOffC);
      for (int s = 0; s < 16; ++s) mma_tf32_ts(tb + kTP1, tb + kTH + s * 8, desc_kmajor(sC, 16384, s), id128, s > 0);
      mma_commit(&bar_mma);
    }
  } else if (tid == 32) {
    // v_new was requested at the start: its copy lands before the CTA can exit, also when
    // aborting
    const bool vn_ok = mbar_wait(&bar_tma2, 0, &abort_flag, p.status, kDevTimeoutTma) || mbar_drain(&bar_tma2, 0);
    if (tma_ok) {
      tc_fence_after();
      const uint32_t id64 = idesc_tf32(128, 64), sVN = smem_u32(sm + kOffVN);
      if (vn_ok && !abort_flag)
        for (int s = 0; s < 16; ++s) mma_tf32_ts(tb + kTP3, tb + kTDH + s * 8, desc_kmajor(sVN, 8192, s), id64, s > 0);
      mma_commit(&bar_mma3);
    }
  }
  // A^T operand of the second product group, built while the first products run (A comes
  // from HBM; nothing before the second group reads it)
  // element (j, i) = A[i][j]; four threads split the 64 rows i of column j = tid % 64.
  {
    const int j = tid & 63, i0 = (tid >> 6) * 16;
    const float* a = p.A + tile * kTileAqk + j;
    float buf[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) buf[e] = a[size_t(i0 + e) * kC];
#pragma unroll
    for (int e = 0; e < 16; ++e) *reinterpret_cast<float*>(sm + kOffAT + sw128_offset(j, i0 + e, kC, 4)) = to_tf32(buf[e]);
  }
  fence_async_smem();
  __syncwarp();
  const bool ok = mbar_wait(&bar_mma, 0, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();
  if (ok) {
    // this thread's tokens t = t0 + e of the 64-token columns
    const int t0 = 32 * hf;
    float r[32];
    // dQt and dKt: token-major rows
    tmem_ld32(tl + kTP1 + t0, r);
    tmem_wait_ld_regs(r);
    store_col_bf16<32>(p.dQt + tile * kTileW + size_t(t0) * kD, r, f);
    // dW^T = -(h dv_new^T): saved token-major (tf32, an MMA operand later) and written back
    // to TMEM as the A operand of A^T dW.
    tmem_ld32(tl + kTP2 + t0, r);
    tmem_wait_ld_regs(r);
    float* dw = p.dW + tile * kTileW + size_t(t0) * kD + f;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      r[e] = to_tf32(-r[e]);
      dw[size_t(e) * kD] = r[e];
    }
    tmem_st32(tl + kTP2 + t0, r);
    // dv_new^T row f (lane f = value column f) as the A operand of A^T dv_new (reuses the first
    // 64 of h's columns), read from the TMA copy of dv_new already in shared memory.
#pragma unroll
    for (int e = 0; e < 32; ++e)
      r[e] = to_tf32(*reinterpret_cast<const float*>(sm + kOffC + sw128_offset(kC + t0 + e, f, 2 * kC, 4)));
    tmem_st32(tl + kTH + t0, r);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && ok && !abort_flag) {
    const uint32_t id64 = idesc_tf32(128, 64);
    const uint32_t sAT = smem_u32(sm + kOffAT);
    // A^T dv_new into h's last 64 columns (dh', P3's operand, may still be being read)
    for (int s = 0; s < 8; ++s) mma_tf32_ts(tb + kTP5, tb + kTP2 + s * 8, desc_kmajor(sAT, 8192, s), id64, s > 0);
    for (int s = 0; s < 8; ++s) mma_tf32_ts(tb + kTH + 64, tb + kTH + s * 8, desc_kmajor(sAT, 8192, s), id64, s > 0);
    mma_commit(&bar_mma);
  }
  __syncwarp();
  // dKt = P3, token-major rows, while the second group runs
  const bool ok3 = ok && mbar_wait(&bar_mma3, 0, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();
  if (ok3) {
    const int t0 = 32 * hf;
    float r[32];
    tmem_ld32(tl + kTP3 + t0, r);
    tmem_wait_ld_regs(r);
    store_col_bf16<32>(p.dKt + tile * kTileW + size_t(t0) * kD, r, f);
  }
  const bool ok2 = ok3 && mbar_wait(&bar_mma, 1, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();
  if (ok2) {
    const int t0 = 32 * hf;
    float r[32];
    tmem_ld32(tl + kTP5 + t0, r);
    tmem_wait_ld_regs(r);
    store_col_bf16<32>(p.dK1 + tile * kTileW + size_t(t0) * kD, r, f);
    tmem_ld32(tl + kTH + 64 + t0, r);
    tmem_wait_ld_regs(r);
    float* v1 = p.dV1 + tile * kTileW + size_t(t0) * kD + f;
#pragma unroll
    for (int e = 0; e < 32; ++e) v1[size_t(e) * kD] = r[e];
  }
  // dgam: per key row (KDA: the two column halves of row f) or summed over the block (GDN).
  if (p.kda) {
    s_dg[tid] = dg;
  } else {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dg += __shfl_xor_sync(0xffffffffu, dg, off);
    if (lane == 0) s_red[warp] = dg;
  }
  tc_fence_before();
  __syncthreads();
  if (p.kda) {
    if (hf == 0) p.dgam[tile * kD + f] = s_dg[f] + s_dg[f + 128];
  } else if (tid == 0) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += s_red[w];
    p.dgam[tile * kD] = sum;
  }
  if (warp == 0) tmem_dealloc(tb, 512);
}

cudaError_t launch_bwd_feat(const CUtensorMap& mVN, const CUtensorMap& mDVN, const CUtensorMap& mdO,
                            const CUtensorMap& mH, const CUtensorMap& mDH, const BwdFeatParams& p, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_bwd_feat, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(unsigned(p.NC) * unsigned(p.hgn));
  k_bwd_feat<<<grid, kThreads, kSmemBytes, s>>>(mVN, mDVN, mdO, mH, mDH, p);
  return cudaGetLastError();
}

}  // namespace gdn
