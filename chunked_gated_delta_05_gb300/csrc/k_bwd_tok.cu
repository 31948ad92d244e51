// Backward, token-major part (scalar gate): the chunk-local adjoint of the prepare step and
// the assembly of the input gradients, one CTA per chunk and head.
//
// Chunk quantities (see the prepare kernel): G = chunk-local cumulative gate, Gam_ij =
// exp(G_i - G_j); k^ = r_k k, q^ = r_q q (L2 norm, r = rsqrt(|x|^2 + 1e-6));
//   L    = strictly_lower(beta_i Gam_ij (k^_i . k^_j)),  A = (I + L)^-1,
//   W    = A K1, K1 = diag(beta exp(G)) k^;   U = A V1, V1 = diag(beta) v;
//   Aqk  = lower(scale Gam_ij (q^_i . k^_j));  Qt = scale diag(exp(G)) q^;
//   Kt   = diag(exp(G_last - G)) k^;           gam = exp(G_last).
// Given dAqk = dO v_new^T, dW, dU = dv_new (feature-major kernel, reverse chain), the
// chain rule through these definitions is:
//   dA   = dW K1^T + dU V1^T,            dL = strictly_lower(-A^T dA A^T)
//   dq^  = (scale dAqk (.) Gam) k^ + scale exp(G) dQt
//   dk^  = (dL beta (.) Gam) k^ + (dL beta (.) Gam)^T k^ + (scale dAqk (.) Gam)^T q^
//          + diag(beta exp(G)) dK1 + diag(exp(G_last - G)) dKt
//   dbeta_i = sum_j dL_ij Gam_ij (k^_i . k^_j) + exp(G_i) (dK1_i . k^_i) + (dV1_i . v_i)
//   dG_i = row_i(P) - col_i(P) + scale exp(G_i)(dQt_i . q^_i) + beta_i exp(G_i)(dK1_i . k^_i)
//          - (dKt_i . Kt_i),   P = dL (.) L + dAqk (.) Aqk,
//   dG_last += sum_i (dKt_i . Kt_i) + gam dgam
//   dg  = reverse cumulative sum of dG within the chunk (g -> G is a cumulative sum)
//   dq  = r_q (dq^ - q^ (q^ . dq^)),  dk likewise   (L2-norm backward)
//   dv  = diag(beta) dV1;  dbeta_logit = dbeta sigmoid'(.) when beta was a logit.
// GB300 mapping: all token x token products are 64-row tcgen05 MMAs (kind::tf32; the raw
// Gram products K K^T and Q K^T are recomputed exactly with kind::f16 on the bf16 tiles), so
// row r of a result sits in TMEM lane 32*(r/16) + r%16 and the 64 threads with lane < 16
// own one token row each. dA is one K=256 product over [dW | dU] and [K1 | V1].
#include "common.cuh"
#include "umma.cuh"

namespace gdn {

namespace {

constexpr int kThreads = 256;   // 8 warps; two threads per TMEM lane (halves of the columns)
constexpr uint32_t kOffQ = 0, kOffK = 16384, kOffV = 32768;   // bf16 [64][128], 2 panels of 8 KB
constexpr uint32_t kR1 = 49152, kR2 = 81920, kR3 = 114688, kR4 = 147456;  // 32 KB regions
constexpr uint32_t kOffDO = 180224;                            // dO bf16 [64][128] (TMA)
constexpr uint32_t kSmemBytes = 196608 + 1024;
// TMEM columns (64-row results)
constexpr uint32_t kTAqk = 0, kTKK = 64, kTQK = 128, kTdA = 192, kTX = 192, kTdL = 192;
constexpr uint32_t kTRq = 0, kTRk = 128;  // reuse after the first products are consumed

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ float bf16_at(const uint8_t* tile, int row, int col) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + sw128_offset(row, col, kC, 2)));
}
__device__ __forceinline__ void put32(uint8_t* tile, int rows, int row, int col, float x) {
  *reinterpret_cast<float*>(tile + sw128_offset(row, col, rows, 4)) = x;
}
// Four consecutive fp32 columns (col % 4 == 0: one 16-byte chunk of the swizzled row).
__device__ __forceinline__ void put32x4(uint8_t* tile, int rows, int row, int col, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(tile + sw128_offset(row, col, rows, 4)) = make_float4(a, b, c, d);
}
// Four consecutive bf16 columns (col % 4 == 0) of a 64-row bf16 tile, as fp32.
__device__ __forceinline__ void bf16x4_at(const uint8_t* tile, int row, int col, float* f) {
  const uint2 u = *reinterpret_cast<const uint2*>(tile + sw128_offset(row, col, kC, 2));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    k_bwd_tok(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdO,
              const __grid_constant__ CUtensorMap mVN, const __grid_constant__ CUtensorMap mDW,
              const __grid_constant__ CUtensorMap mDVN, const BwdTokParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1k(smem_raw);
  __shared__ uint64_t bar_tma, bar_tma2, bar_mma;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;
  __shared__ float s_G[kC], s_G2[kC], s_rq[kC], s_rk[kC], s_b[kC], s_e1[kC], s_dG[kC], s_db[kC], s_P[kC][kC + 1];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // heads fastest: the CTAs in flight share token rows of the inputs and gradients
  const int c = int(blockIdx.x / p.hgn), h = int(blockIdx.x % p.hgn) + p.hg0, H = p.H;
  const size_t tile = size_t(c) * H + h;
  const ChunkEntry ch = chunk_entry(p.chunks, c, p.dense_T);
  const int len = ch.y;
  const int wq = warp & 3, half = warp >> 2;   // TMEM lane quadrant; which half of the columns
  const bool owner = lane < 16;                // owns token row rr of every 64-row MMA result
  const int rr = 16 * wq + (lane & 15);
  const float scale = p.scale;
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sK = sm + kOffK;
  uint8_t* sV = sm + kOffV;

  if (warp == 0) tmem_alloc(&tslot, 256);
  if (tid == 0) {
    // The barriers are this thread's alone until the block barrier below, so the loads start
    // right after their initialisation. First group (q, k, v, dO, v_new) feeds the first
    // products; dW, dU arrive on their own barrier and are first read by the dA product.
    abort_flag = 0;
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_tma2, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    mbar_expect_tx(&bar_tma, 4u * 16384u + 32768u);
    mbar_expect_tx(&bar_tma2, 2u * 32768u);
    for (int pp = 0; pp < 4; ++pp) {  // chunk-tile rows: no wait for the chunk table
      tma_load_2d(sm + kR2 + pp * 8192, &mVN, pp * 32, int(tile) * kC, &bar_tma);
      tma_load_2d(sm + kR3 + pp * 8192, &mDW, pp * 32, int(tile) * kC, &bar_tma2);
      tma_load_2d(sm + kR4 + pp * 8192, &mDVN, pp * 32, int(tile) * kC, &bar_tma2);
    }
    for (int pp = 0; pp < 2; ++pp) {
      const int x = h * kD + 64 * pp, xqk = (h / p.qk_group) * kD + 64 * pp;
      tma_load_2d(sQ + pp * 8192, &mq, xqk, ch.x, &bar_tma);
      tma_load_2d(sK + pp * 8192, &mk, xqk, ch.x, &bar_tma);
      tma_load_2d(sV + pp * 8192, &mv, x, ch.x, &bar_tma);
      tma_load_2d(sm + kOffDO + pp * 8192, &mdO, x, ch.x, &bar_tma);
    }
    // inputs of the later phases: start their trip from HBM now
    const size_t rows = tile * kTileW;
    prefetch_l2(p.A + tile * kTileAqk, 4u * kTileAqk);
    prefetch_l2(p.dQt + rows, 2u * kTileW);
    prefetch_l2(p.dKt + rows, 2u * kTileW);
    prefetch_l2(p.dK1 + rows, 2u * kTileW);
    prefetch_l2(p.dV1 + rows, 4u * kTileW);
  }
  if (tid < kC) {
    // requested before the chunk length is known, masked after
    const float G = p.Gc[tile * kC + tid], rq = p.rq[tile * kC + tid], rk = p.rk[tile * kC + tid],
                b = p.beff[tile * kC + tid];
    const bool ok = tid < len;
    s_G[tid] = G;
    s_G2[tid] = G * kLog2e;  // exp(G_i - G_j) = exp2(G2_i - G2_j) in the pair loop
    s_rq[tid] = ok ? rq : 0.f;
    s_rk[tid] = ok ? rk : 0.f;
    s_b[tid] = ok ? b : 0.f;
    s_e1[tid] = ok ? b * expf(G) * rk : 0.f;   // the row scale of K1
    s_dG[tid] = 0.f;
    s_db[tid] = 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  const uint32_t tl = tb + tmem_lane_base(warp);
  const float Glast = s_G[len - 1];
  const bool tma_ok = mbar_wait(&bar_tma, 0, &abort_flag, p.status, kDevTimeoutTma);
  // A full chunk has no rows to clear, so its exact Gram products K K^T and Q K^T (raw bf16
  // tiles) go out now and run under the dO conversion; a ragged chunk issues them with dAqk.
  const bool early_gram = len == kC;
  if (tid == 0 && tma_ok && early_gram) {
    tc_fence_after();
    const uint32_t id_bf = idesc_bf16(64, 64), q0 = smem_u32(sQ), k0 = smem_u32(sK);
    for (int s = 0; s < 8; ++s) mma_bf16_ss(tb + kTKK, desc_kmajor(k0, 8192, s), desc_kmajor(k0, 8192, s), id_bf, s > 0);
    for (int s = 0; s < 8; ++s) mma_bf16_ss(tb + kTQK, desc_kmajor(q0, 8192, s), desc_kmajor(k0, 8192, s), id_bf, s > 0);
  }
  // dO as a 64-row tf32 operand [i][v] (rows past the chunk are zero): thread row tid / 4,
  // 32 columns, eight per 16-byte read of the bf16 tile.
  {
    const int t = tid >> 2, cq = 32 * (tid & 3);
    const bool in = t < len;
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
      const int col = cq + 8 * c8;
      float f[8];
      if (in) {
        const uint4 u = *reinterpret_cast<const uint4*>(sm + kOffDO + sw128_offset(t, col, kC, 2));
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(b2[e]);
          f[2 * e] = x.x;
          f[2 * e + 1] = x.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = 0.f;
      }
      put32x4(sm + kR1, kC, t, col, f[0], f[1], f[2], f[3]);
      put32x4(sm + kR1, kC, t, col + 4, f[4], f[5], f[6], f[7]);
    }
  }
  // Rows of q, k, v past the chunk belong to the next document (or are zero): clear them so
  // the exact Gram products below see zeros there.
  if (tid >= len && tid < kC) {
    for (int c16 = 0; c16 < 16; ++c16) {
      const uint32_t off = sw128_offset(tid, c16 * 8, kC, 2);
      *reinterpret_cast<uint4*>(sQ + off) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sK + off) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sV + off) = make_uint4(0, 0, 0, 0);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- products 1: dAqk = dO v_new^T, K K^T, Q K^T
  if (tid == 0 && tma_ok) {
    const uint32_t id_tf = idesc_tf32(64, 64), id_bf = idesc_bf16(64, 64);
    const uint32_t r1 = smem_u32(sm + kR1), r2 = smem_u32(sm + kR2);
    const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK);
    for (int s = 0; s < 16; ++s) mma_tf32_ss(tb + kTAqk, desc_kmajor(r1, 8192, s), desc_kmajor(r2, 8192, s), id_tf, s > 0);
    if (!early_gram) {
      for (int s = 0; s < 8; ++s) mma_bf16_ss(tb + kTKK, desc_kmajor(k0, 8192, s), desc_kmajor(k0, 8192, s), id_bf, s > 0);
      for (int s = 0; s < 8; ++s) mma_bf16_ss(tb + kTQK, desc_kmajor(q0, 8192, s), desc_kmajor(k0, 8192, s), id_bf, s > 0);
    }
    mma_commit(&bar_mma);  // covers the early Gram products too (same issuing thread)
  }
  __syncwarp();
  bool ok = tma_ok && mbar_wait(&bar_mma, 0, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();
  // ---- K1 = diag(beta exp(G) r_k) k and V1 = diag(beta) v as 64-row operands [j][d]
  // (a warp converts one row per step: lane l takes columns 4l..4l+3, one 16-byte chunk)
  {
    const int c0 = 4 * lane;
#pragma unroll 2
    for (int j = warp; j < kC; j += 8) {
      const float s1 = s_e1[j], s2 = s_b[j];
      float kf[4], vf[4];
      bf16x4_at(sK, j, c0, kf);
      bf16x4_at(sV, j, c0, vf);
      put32x4(sm + kR1, kC, j, c0, to_tf32(s1 * kf[0]), to_tf32(s1 * kf[1]), to_tf32(s1 * kf[2]), to_tf32(s1 * kf[3]));
      put32x4(sm + kR2, kC, j, c0, to_tf32(s2 * vf[0]), to_tf32(s2 * vf[1]), to_tf32(s2 * vf[2]), to_tf32(s2 * vf[3]));
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // ---- product 2: dA = [dW | dU] [K1 | V1]^T  (K = 256)
  if (tid == 0 && ok) ok = mbar_wait(&bar_tma2, 0, &abort_flag, p.status, kDevTimeoutTma);
  if (tid == 0 && ok) {
    const uint32_t id_tf = idesc_tf32(64, 64);
    const uint32_t r1 = smem_u32(sm + kR1), r2 = smem_u32(sm + kR2), r3 = smem_u32(sm + kR3), r4 = smem_u32(sm + kR4);
    for (int s = 0; s < 16; ++s) mma_tf32_ss(tb + kTdA, desc_kmajor(r3, 8192, s), desc_kmajor(r1, 8192, s), id_tf, s > 0);
    for (int s = 0; s < 16; ++s) mma_tf32_ss(tb + kTdA, desc_kmajor(r4, 8192, s), desc_kmajor(r2, 8192, s), id_tf, true);
    mma_commit(&bar_mma);
  }
  __syncwarp();
  // A [i][j] (thread: column j, 16 rows i) is requested now, so that its trip from L2 overlaps
  // the products
  float abuf[16];
  {
    const float* a = p.A + tile * kTileAqk + (tid & 63);
    const int i0 = 16 * (tid >> 6);
#pragma unroll
    for (int e = 0; e < 16; ++e) abuf[e] = a[size_t(i0 + e) * kC];
  }
  ok = ok && mbar_wait(&bar_mma, 1, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();
  // ---- dL = -A^T dA A^T: X = A^T dA, then X A^T.
  // Operands (64x64 tf32, 16 KB each): AT [j][i] (A op), dAT [m][i] (B op), A [l][m] (B op), X.
  uint8_t* sAT = sm + kR3;
  uint8_t* sdAT = sm + kR3 + 16384;
  uint8_t* sA = sm + kR4;
  uint8_t* sX = sm + kR4 + 16384;
  // a 64-row result read with the 16x64b shape: lane t holds row ri of the warp's 16 at
  // columns cj + 2 r (all 32 lanes busy)
  const int ri = 16 * wq + (lane >> 2) + 8 * (lane & 1), cj = 32 * half + ((lane >> 1) & 1);
  {
    float r[16];
    tmem_ld16x64b_x16(tl + kTdA + 32 * half, r);
    tmem_wait_ld_regs(r);
#pragma unroll
    for (int m = 0; m < 16; ++m) put32(sdAT, kC, cj + 2 * m, ri, to_tf32(r[m]));
    {
      // A [i][j] read once, coalesced (thread: column j, 16 rows i), into both operands: A^T
      // (row j, four consecutive i per 16-byte chunk) and A (row i, column j)
      const int j = tid & 63, i0 = 16 * (tid >> 6);
      float buf[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) buf[e] = to_tf32(abuf[e]);
#pragma unroll
      for (int e = 0; e < 16; e += 4) put32x4(sAT, kC, j, i0 + e, buf[e], buf[e + 1], buf[e + 2], buf[e + 3]);
#pragma unroll
      for (int e = 0; e < 16; ++e) put32(sA, kC, i0 + e, j, buf[e]);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && ok) {
    const uint32_t id_tf = idesc_tf32(64, 64);
    for (int s = 0; s < 8; ++s)
      mma_tf32_ss(tb + kTX, desc_kmajor(smem_u32(sAT), 8192, s), desc_kmajor(smem_u32(sdAT), 8192, s), id_tf, s > 0);
    mma_commit(&bar_mma);
  }
  __syncwarp();
  ok = ok && mbar_wait(&bar_mma, 0, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();
  {
    float r[16];
    tmem_ld16x64b_x16(tl + kTX + 32 * half, r);
    tmem_wait_ld_regs(r);
#pragma unroll
    for (int m = 0; m < 16; ++m) put32(sX, kC, ri, cj + 2 * m, to_tf32(r[m]));
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && ok) {
    const uint32_t id_tf = idesc_tf32(64, 64);
    for (int s = 0; s < 8; ++s)
      mma_tf32_ss(tb + kTdL, desc_kmajor(smem_u32(sX), 8192, s), desc_kmajor(smem_u32(sA), 8192, s), id_tf, s > 0);
    mma_commit(&bar_mma);
  }
  __syncwarp();
  ok = ok && mbar_wait(&bar_mma, 1, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();

  // ---- elementwise on token pairs: row owner i holds row i of dL', dAqk, KK, QK.
  // A operands for the last products: E1 [i][j], E2^T [j][i], Nq [i][j], Nk^T [j][i];
  // B operands: k^T [d][j], q^T [d][i] (raw tiles, tf32).
  uint8_t* sE1 = sm + kR1;
  uint8_t* sE2T = sm + kR1 + 16384;
  uint8_t* sNq = sm + kR2;
  uint8_t* sNkT = sm + kR2 + 16384;
  uint8_t* sKT = sm + kR3;   // [128][64]: 2 panels x 128 rows
  uint8_t* sQT = sm + kR4;
  {
    // the 16x64b TMEM shape spreads a quadrant's 16 rows over all 32 lanes: lane t holds row
    // (t >> 2) + 8 (t & 1) at columns ((t >> 1) & 1) + 2 r, so a row's 32 columns of this half
    // sit on the lane pair (t, t ^ 2)
    const int i = ri;
    const int jb = cj;
    const bool vi = i < len;
    const float Gi2 = s_G2[i], bi = s_b[i], rki = s_rk[i], rqi = s_rq[i];
    float rowP = 0.f, dbi = 0.f;
    {
      float dl[16], nn[16], kk[16], qk[16];
      tmem_ld16x64b_x16(tl + kTdL + 32 * half, dl);
      tmem_ld16x64b_x16(tl + kTAqk + 32 * half, nn);
      tmem_ld16x64b_x16(tl + kTKK + 32 * half, kk);
      tmem_ld16x64b_x16(tl + kTQK + 32 * half, qk);
      tmem_wait_ld_regs(dl);
      tmem_wait_ld_regs(nn);
      tmem_wait_ld_regs(kk);
      tmem_wait_ld_regs(qk);
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int j = jb + 2 * jj;
        const float gam = (j <= i && vi) ? exp2f(Gi2 - s_G2[j]) : 0.f;
        const float D = (j < i && vi) ? -dl[jj] : 0.f;                 // dL_ij
        const float N = (j <= i && vi) ? nn[jj] : 0.f;                 // dAqk_ij
        const float rkj = s_rk[j];
        const float Lij = bi * rki * rkj * kk[jj] * gam;
        const float Aij = scale * rqi * rkj * qk[jj] * gam;
        const float P = D * Lij + N * Aij;
        rowP += P;
        s_P[i][j] = P;
        dbi = fmaf(D * rki * rkj * kk[jj], gam, dbi);
        const float e = D * bi * gam;
        put32(sE1, kC, i, j, to_tf32(e * rkj));
        put32(sE2T, kC, j, i, to_tf32(e * rki));
        const float nq = scale * N * gam;
        put32(sNq, kC, i, j, to_tf32(nq * rkj));
        put32(sNkT, kC, j, i, to_tf32(nq * rqi));
      }
    }
    // the row's two lanes combine, then one adds the half-row sums
    rowP += __shfl_xor_sync(0xffffffffu, rowP, 2);
    dbi += __shfl_xor_sync(0xffffffffu, dbi, 2);
    if (((lane >> 1) & 1) == 0) {
      atomicAdd(&s_dG[i], rowP);
      atomicAdd(&s_db[i], dbi);
    }
  }
  // transposed raw tiles k^T [d][j], q^T [d][i] (zero past the chunk: cleared above)
  // (thread: row d, four consecutive token columns per step, one 16-byte chunk)
  {
    const int d = tid & 127;
#pragma unroll 2
    for (int j = 4 * half; j < kC; j += 8) {
      put32x4(sKT, kD, d, j, to_tf32(bf16_at(sK, j, d)), to_tf32(bf16_at(sK, j + 1, d)),
              to_tf32(bf16_at(sK, j + 2, d)), to_tf32(bf16_at(sK, j + 3, d)));
      put32x4(sQT, kD, d, j, to_tf32(bf16_at(sQ, j, d)), to_tf32(bf16_at(sQ, j + 1, d)),
              to_tf32(bf16_at(sQ, j + 2, d)), to_tf32(bf16_at(sQ, j + 3, d)));
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // ---- products 4: dq^ part = Nq k^T^T (rows i); dk^ part = E1 k + E2^T k + Nk^T q (rows)
  if (tid == 0 && ok) {
    const uint32_t id = idesc_tf32(64, 128);
    const uint32_t kt = smem_u32(sKT), qt = smem_u32(sQT);
    for (int s = 0; s < 8; ++s) mma_tf32_ss(tb + kTRq, desc_kmajor(smem_u32(sNq), 8192, s), desc_kmajor(kt, 16384, s), id, s > 0);
    for (int s = 0; s < 8; ++s) mma_tf32_ss(tb + kTRk, desc_kmajor(smem_u32(sE1), 8192, s), desc_kmajor(kt, 16384, s), id, s > 0);
    for (int s = 0; s < 8; ++s) mma_tf32_ss(tb + kTRk, desc_kmajor(smem_u32(sE2T), 8192, s), desc_kmajor(kt, 16384, s), id, true);
    for (int s = 0; s < 8; ++s) mma_tf32_ss(tb + kTRk, desc_kmajor(smem_u32(sNkT), 8192, s), desc_kmajor(qt, 16384, s), id, true);
    mma_commit(&bar_mma);
  }
  // column sums of P while the products run
  if (tid < kC) {
    float col = 0.f;
#pragma unroll 8
    for (int i = 0; i < kC; ++i) col += s_P[i][tid];
    s_dG[tid] -= col;
  }
  __syncwarp();
  ok = ok && mbar_wait(&bar_mma, 0, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();

  // ---- per-token assembly. Owner threads stage their rows of the two last products from
  // TMEM into padded shared rows; then each warp takes whole token rows (lane l: columns
  // 4l..4l+3) with coalesced loads of the intermediates (dV1 fp32; dQt, dKt, dK1 bf16) and
  // shuffle-reduced dots.
  constexpr int kPad = 132;                                  // padded row stride (floats)
  float* sRq = reinterpret_cast<float*>(sm + kR1);           // [64][132]
  float* sRk = sRq + kC * kPad;                              // [64][132]
  if (ok) {
    {
      const int which = half;
      float* dst = (which == 0 ? sRq : sRk) + rr * kPad;
      const uint32_t col = which == 0 ? kTRq : kTRk;
      for (int g4 = 0; g4 < 4; ++g4) {
        float r[32];
        tmem_ld32(tl + col + 32 * g4, r);
        tmem_wait_ld_regs(r);
        if (owner) {
          float4* d4 = reinterpret_cast<float4*>(dst + 32 * g4);
#pragma unroll
          for (int e = 0; e < 8; ++e) d4[e] = make_float4(r[4 * e], r[4 * e + 1], r[4 * e + 2], r[4 * e + 3]);
        }
      }
    }
  }
  __syncthreads();
  if (ok) {
    // eight lanes per token row (lane l8 of the group: features 32 m + 4 l8 + e, m, e < 4, so
    // the group's loads and stores of one m are 128 contiguous bytes), four rows per warp at a
    // time, so each 3-level butterfly reduces four rows' dots at once; warp w takes rows
    // 8 w .. 8 w + 7. Lanes of rows past the chunk run with zeros and store nothing.
    const size_t rowbase = tile * kTileW;
    const int g = lane >> 3, l8 = lane & 7, d0 = 4 * l8;
    const int Hk = H / p.qk_group;
    auto sum8 = [](float x) {
      x += __shfl_xor_sync(0xffffffffu, x, 4);
      x += __shfl_xor_sync(0xffffffffu, x, 2);
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      return x;
    };
    // element 4 m + e of a lane's 16 is feature d0 + 32 m + e
    auto bf16x16 = [&](const uint8_t* tile16, int t, float* f) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint2 u = *reinterpret_cast<const uint2*>(tile16 + sw128_offset(t, d0 + 32 * m, kC, 2));
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
        f[4 * m] = a.x; f[4 * m + 1] = a.y; f[4 * m + 2] = b.x; f[4 * m + 3] = b.y;
      }
    };
    auto store16 = [&](__nv_bfloat16* dst, const float* x) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        __nv_bfloat162 a = __floats2bfloat162_rn(x[4 * m], x[4 * m + 1]), b = __floats2bfloat162_rn(x[4 * m + 2], x[4 * m + 3]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&a);
        u.y = *reinterpret_cast<uint32_t*>(&b);
        *reinterpret_cast<uint2*>(dst + 32 * m) = u;
      }
    };
    auto load16 = [&](const float* src, bool v, float* f) {   // read-only for this kernel
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float4 x = v ? __ldg(reinterpret_cast<const float4*>(src + 32 * m)) : make_float4(0.f, 0.f, 0.f, 0.f);
        f[4 * m] = x.x; f[4 * m + 1] = x.y; f[4 * m + 2] = x.z; f[4 * m + 3] = x.w;
      }
    };
    auto load16h = [&](const __nv_bfloat16* src, bool v, float* f) {   // bf16 tiles, read-only
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float4 x = v ? ldg_bf16x4(src + 32 * m) : make_float4(0.f, 0.f, 0.f, 0.f);
        f[4 * m] = x.x; f[4 * m + 1] = x.y; f[4 * m + 2] = x.z; f[4 * m + 3] = x.w;
      }
    };
    auto smem16 = [&](const float* src, float* f) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float4 x = *reinterpret_cast<const float4*>(src + 32 * m);
        f[4 * m] = x.x; f[4 * m + 1] = x.y; f[4 * m + 2] = x.z; f[4 * m + 3] = x.w;
      }
    };
#pragma unroll 1
    for (int it = 0; it < 2; ++it) {
      const int t = 8 * warp + 4 * it + g;
      const bool valid = t < len;
      const int tt = valid ? t : 0;
      const size_t ro = rowbase + size_t(tt) * kD + d0;
      float dqt[16], k1v[16], ktv[16], v1v[16];
      load16h(p.dQt + ro, valid, dqt);
      load16h(p.dK1 + ro, valid, k1v);
      load16h(p.dKt + ro, valid, ktv);
      load16(p.dV1 + ro, valid, v1v);
      const float Gt = s_G[tt], rqt = s_rq[tt], rkt = s_rk[tt], bt = s_b[tt];
      const float eG = expf(Gt), eL = expf(Glast - Gt);
      const size_t orow = (size_t(ch.x + tt) * H + h) * kD + d0;
      const size_t oqk = (size_t(ch.x + tt) * Hk + h / p.qk_group) * kD + d0;
      float x[16];
      // dq
      float dot = 0.f, qdq = 0.f;
      {
        float qv[16], a[16], rq[16];
        bf16x16(sQ, tt, qv);
        smem16(sRq + tt * kPad + d0, rq);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float qh = rqt * qv[e];
          a[e] = fmaf(scale * eG, dqt[e], rq[e]);
          dot = fmaf(a[e], qh, dot);
          qdq = fmaf(dqt[e], qh, qdq);
        }
        dot = sum8(dot);
        qdq = sum8(qdq);
        if (!p.l2norm) dot = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = rqt * (a[e] - rqt * qv[e] * dot);
      }
      if (valid) {
        if (p.dq32) {
#pragma unroll
          for (int m = 0; m < 4; ++m)
            *reinterpret_cast<float4*>(p.dq32 + orow + 32 * m) = make_float4(x[4 * m], x[4 * m + 1], x[4 * m + 2], x[4 * m + 3]);
        } else {
          store16(p.dq + oqk, x);
        }
      }
      // dk
      float kdot = 0.f, k1k = 0.f, ktk = 0.f;
      {
        float kv[16], a[16], rk[16];
        bf16x16(sK, tt, kv);
        smem16(sRk + tt * kPad + d0, rk);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float kh = rkt * kv[e];
          a[e] = rk[e] + bt * eG * k1v[e] + eL * ktv[e];
          kdot = fmaf(a[e], kh, kdot);
          k1k = fmaf(k1v[e], kh, k1k);
          ktk = fmaf(ktv[e], kh, ktk);
        }
        kdot = sum8(kdot);
        k1k = sum8(k1k);
        ktk = sum8(ktk);
        if (!p.l2norm) kdot = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = rkt * (a[e] - rkt * kv[e] * kdot);
      }
      if (valid) {
        if (p.dk32) {
#pragma unroll
          for (int m = 0; m < 4; ++m)
            *reinterpret_cast<float4*>(p.dk32 + orow + 32 * m) = make_float4(x[4 * m], x[4 * m + 1], x[4 * m + 2], x[4 * m + 3]);
        } else {
          store16(p.dk + oqk, x);
        }
      }
      // dv and the v part of dbeta
      float vv = 0.f;
      {
        float vvv[16];
        bf16x16(sV, tt, vvv);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          vv = fmaf(v1v[e], vvv[e], vv);
          x[e] = bt * v1v[e];
        }
        vv = sum8(vv);
      }
      if (valid) {
        store16(p.dv + orow, x);
        if (l8 == 0) {
          s_dG[t] += scale * eG * qdq + bt * eG * k1k - eL * ktk;
          s_db[t] += eG * k1k + vv;
          s_P[t][0] = eL * ktk;   // this row's share of dG_last (column 0 of P is free now)
        }
      }
    }
  }
  __syncthreads();
  if (warp == 0 && ok) {
    // gate: G_last collects the end-decay terms; the reverse cumulative sum gives dg. Lane l
    // holds rows 2 l and 2 l + 1; a suffix scan over the lanes replaces the serial loop.
    const int t0 = 2 * lane, t1 = 2 * lane + 1;
    float base = (t0 < len ? s_P[t0][0] : 0.f) + (t1 < len ? s_P[t1][0] : 0.f);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) base += __shfl_xor_sync(0xffffffffu, base, off);
    base += expf(Glast) * p.dgam[tile * kD];
    const float a0 = t0 < len ? s_dG[t0] : 0.f, a1 = t1 < len ? s_dG[t1] : 0.f;
    const float pair = a0 + a1;
    float suf = pair;   // inclusive suffix sum over lanes >= l
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, suf, off);
      if (lane + off < 32) suf += y;
    }
    const float after = base + suf - pair;   // rows past 2 l + 1
    if (t1 < len) s_dG[t1] = after + a1;
    if (t0 < len) s_dG[t0] = after + a1 + a0;
  }
  __syncthreads();
  if (tid < len && ok) {
    const size_t o = size_t(ch.x + tid) * H + h;
    // a gate below the floor was clamped in the forward: its gradient is 0
    p.dg[o] = p.g[o] < kGateFloor ? 0.f : s_dG[tid];
    float db = s_db[tid];
    if (p.beta_sigmoid) db *= s_b[tid] * (1.f - s_b[tid]);
    p.dbeta[o] = __float2bfloat16_rn(db);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 256);
}

cudaError_t launch_bwd_tok(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdO,
                           const CUtensorMap& mVN, const CUtensorMap& mDW, const CUtensorMap& mDVN, const BwdTokParams& p,
                           cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_bwd_tok, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(unsigned(p.NC) * unsigned(p.hgn));
  k_bwd_tok<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, mdO, mVN, mDW, mDVN, p);
  return cudaGetLastError();
}

}  // namespace gdn
