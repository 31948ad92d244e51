// Backward, token-major part for the per-channel gate (Kimi Delta Attention), one CTA per
// chunk and head.
//
// Same chunk quantities as the scalar-gate kernel, with every decay per key channel c:
//   L_ij   = beta_i sum_c k^_ic k^_jc Gam_ijc,  Aqk_ij = scale sum_c q^_ic k^_jc Gam_ijc,
//   Gam_ijc = exp(G_ic - G_jc);  K1_jc = beta_j exp(G_jc) k^_jc;  Qt_ic = scale exp(G_ic) q^_ic;
//   Kt_ic = exp(G_last,c - G_ic) k^_ic;  gam_c = exp(G_last,c).
// With D = dL (strictly lower) and N = dAqk (lower), the decayed pair sums
//   X1_ic = sum_{j<i} D_ij k^_jc Gam_ijc          Y1_ic = scale sum_{j<=i} N_ij k^_jc Gam_ijc
//   Z_jc  = sum_{i>j} beta_i D_ij k^_ic Gam_ijc + scale sum_{i>=j} N_ij q^_ic Gam_ijc
// give
//   dk^ = beta X1 + Z + diag(beta) exp(G) (.) dK1 + exp(G_last - G) (.) dKt
//   dq^ = Y1 + scale exp(G) (.) dQt
//   dG  = beta k^ (.) X1 + q^ (.) Y1 - k^ (.) Z + beta exp(G) (.) dK1 (.) k^
//         + scale exp(G) (.) dQt (.) q^ - exp(G_last - G) (.) dKt (.) k^       (per channel)
//   dG_last,c += sum_i exp(G_last,c - G_ic) dKt_ic k^_ic + gam_c dgam_c
//   dbeta_i = sum_c k^_ic X1_ic + sum_c exp(G_ic) dK1_ic k^_ic + sum_c dV1_ic v_ic
//   dg = reverse cumulative sum of dG over the chunk's tokens, per channel.
// GB300 mapping: dAqk, dA = [dW | dU][K1 | V1]^T, A^T dA and (A^T dA) A^T are 64-row
// tcgen05 MMAs (kind::tf32) as in the scalar-gate kernel. The decayed pair sums are tensor-core
// products too: each pair's decay factors through the reference row of the later token's
// 16-row block into two bounded per-channel factors (the prepare kernel's Gram factorisation),
// and two rounds of 128-lane products with the channels on the accumulator lanes give X1, Y1
// and Z; the CUDA cores apply the row factors and assemble the gradients.
#include "common.cuh"
#include "umma.cuh"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kP = kD + 1;                                   // padded row stride (floats)
constexpr uint32_t kOffQ = 0, kOffK = 16384, kOffV = 32768;  // bf16 [64][128]
constexpr uint32_t kOffG = 49152;                            // G * log2(e), fp32 [64][129]
constexpr uint32_t kR1 = 83968, kR2 = 116736, kR3 = 149504, kR4 = 182272;  // 32 KB each
constexpr uint32_t kSmemBytes = kR4 + 32768 + 1024;
constexpr uint32_t kTAqk = 0, kTdA = 64, kTX = 128;  // 64-row products
constexpr uint32_t kTXY = 0, kTV = 256;              // pair-sum products (channels on the lanes)

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}
__device__ __forceinline__ float bf16_at(const uint8_t* tile, int row, int col) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + sw128_offset(row, col, kC, 2)));
}
// Four consecutive bf16 columns (col % 4 == 0) of a 64-row bf16 tile, as fp32.
__device__ __forceinline__ void bf16x4_at(const uint8_t* tile, int row, int col, float* f) {
  const uint2 u = *reinterpret_cast<const uint2*>(tile + sw128_offset(row, col, kC, 2));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}
__device__ __forceinline__ uint2 pack_bf16x4(const float* x) {
  __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  return u;
}
__device__ __forceinline__ void put32(uint8_t* tile, int rows, int row, int col, float x) {
  *reinterpret_cast<float*>(tile + sw128_offset(row, col, rows, 4)) = x;
}
// Four consecutive fp32 columns (col % 4 == 0: one 16-byte chunk of the swizzled row).
__device__ __forceinline__ void put32x4(uint8_t* tile, int rows, int row, int col, const float* x) {
  *reinterpret_cast<float4*>(tile + sw128_offset(row, col, rows, 4)) = make_float4(x[0], x[1], x[2], x[3]);
}


}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    k_bwd_tok_kda(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                  const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mVN,
                  const __grid_constant__ CUtensorMap mDW, const __grid_constant__ CUtensorMap mDVN,
                  const __grid_constant__ CUtensorMap mdO, const BwdTokParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1k(smem_raw);
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sK = sm + kOffK;
  uint8_t* sV = sm + kOffV;
  float* sG2 = reinterpret_cast<float*>(sm + kOffG);
  __shared__ uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;
  __shared__ float s_rq[kC], s_rk[kC], s_b[kC];
  // per-token sums over the channels: the pair sums' share of dbeta, one partial per group of
  // 32 channels (warp % 4), added in a fixed order so that the result does not depend on warp
  // scheduling; the assembly's sums (one warp reduction per token row)
  __shared__ float s_dba[1][kC];
  __shared__ __align__(16) float s_glw[kThreads / 32][kD];  // each warp's dG_last shares

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wq = warp & 3, half = warp >> 2;
  // heads fastest: the CTAs in flight share token rows of the inputs and gradients
  const int c_idx = int(blockIdx.x / p.hgn), h = int(blockIdx.x % p.hgn) + p.hg0, H = p.H;
  const size_t tile = size_t(c_idx) * H + h;
  const ChunkEntry ch = chunk_entry(p.chunks, c_idx, p.dense_T);
  const int len = ch.y;
  const bool owner = lane < 16;
  const int rr = 16 * wq + (lane & 15);
  const float scale = p.scale;
  const int cc = tid & 127;   // channel handled in the CUDA-core phases
  const float dgam_c = p.dgam[tile * kD + cc];  // requested now, used by the last phase

  if (warp == 0) tmem_alloc(&tslot, 512);
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  if (tid < kC) {
    const bool ok = tid < len;
    s_rq[tid] = ok ? p.rq[tile * kC + tid] : 0.f;
    s_rk[tid] = ok ? p.rk[tile * kC + tid] : 0.f;
    s_b[tid] = ok ? p.beff[tile * kC + tid] : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  const uint32_t tl = tb + tmem_lane_base(warp);
  if (tid == 0) {
    // q, k, v, v_new, dW, dU; the chunk's G tile (bulk copy into R1) and dO (bf16, into the G
    // area) for the staging below
    mbar_expect_tx(&bar_tma, 4u * 16384u + 4u * 32768u);
    bulk_load(sm + kR1, p.Gc + tile * kC * kD, 32768u, &bar_tma);
    for (int pp = 0; pp < 2; ++pp) tma_load_2d(sm + kOffG + pp * 8192, &mdO, h * kD + 64 * pp, ch.x, &bar_tma);
    for (int pp = 0; pp < 2; ++pp) {
      const int x = h * kD + 64 * pp, xqk = (h / p.qk_group) * kD + 64 * pp;
      tma_load_2d(sQ + pp * 8192, &mq, xqk, ch.x, &bar_tma);
      tma_load_2d(sK + pp * 8192, &mk, xqk, ch.x, &bar_tma);
      tma_load_2d(sV + pp * 8192, &mv, x, ch.x, &bar_tma);
    }
    for (int pp = 0; pp < 4; ++pp) {
      tma_load_2d(sm + kR2 + pp * 8192, &mVN, pp * 32, int(tile) * kC, &bar_tma);
      tma_load_2d(sm + kR3 + pp * 8192, &mDW, pp * 32, int(tile) * kC, &bar_tma);
      tma_load_2d(sm + kR4 + pp * 8192, &mDVN, pp * 32, int(tile) * kC, &bar_tma);
    }
    // inputs of the later phases (the inverse, the assembly's gradient tiles): start their
    // trip from HBM now
    const size_t rows = tile * kTileW;
    prefetch_l2(p.A + tile * kTileAqk, 4u * kTileAqk);
    prefetch_l2(p.dQt + rows, 2u * kTileW);
    prefetch_l2(p.dKt + rows, 2u * kTileW);
    prefetch_l2(p.dK1 + rows, 2u * kTileW);
    prefetch_l2(p.dV1 + rows, 4u * kTileW);
  }
  // G (scaled to log2 units) and dO as a 64-row tf32 operand; rows past the chunk are zero.
  // Both arrived with the other copies (G in R1, dO in the G area): each thread reads its
  // values into registers and, once every thread has, writes them to their places.
  const bool tma_ok = mbar_wait(&bar_tma, 0, &abort_flag, p.status, kDevTimeoutTma);
  {
    const int t0 = 32 * half;
    const float* gt = reinterpret_cast<const float*>(sm + kR1);
    float bg[32], bo[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      bg[e] = gt[(t0 + e) * kD + cc];
      bo[e] = (t0 + e < len) ? bf16_at(sm + kOffG, t0 + e, cc) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      sG2[(t0 + e) * kP + cc] = bg[e] * kLog2e;
      put32(sm + kR1, kC, t0 + e, cc, bo[e]);
    }
  }
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
  // ---- dAqk = dO v_new^T
  if (tid == 0 && tma_ok) {
    const uint32_t id = idesc_tf32(64, 64);
    const uint32_t r1 = smem_u32(sm + kR1), r2 = smem_u32(sm + kR2);
    for (int s = 0; s < 16; ++s) mma_tf32_ss(tb + kTAqk, desc_kmajor(r1, 8192, s), desc_kmajor(r2, 8192, s), id, s > 0);
    mma_commit(&bar_mma);
  }
  __syncwarp();
  bool ok = tma_ok && mbar_wait(&bar_mma, 0, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();
  // ---- K1 = beta r_k exp(G) (.) k and V1 = beta v as 64-row operands [j][c]: each warp takes
  // whole rows, lane l channels 4l .. 4l+3 (one 16-byte chunk of each swizzled row)
  {
    const int c4 = 4 * lane;
    for (int j = warp; j < kC; j += kThreads / 32) {
      const float s1 = s_b[j] * s_rk[j], s2 = s_b[j];
      float kv[4], vv[4], k1[4];
      bf16x4_at(sK, j, c4, kv);
      bf16x4_at(sV, j, c4, vv);
#pragma unroll
      for (int e = 0; e < 4; ++e) k1[e] = to_tf32(s1 * exp2f(sG2[j * kP + c4 + e]) * kv[e]);
      *reinterpret_cast<float4*>(sm + kR1 + sw128_offset(j, c4, kC, 4)) = make_float4(k1[0], k1[1], k1[2], k1[3]);
      *reinterpret_cast<float4*>(sm + kR2 + sw128_offset(j, c4, kC, 4)) =
          make_float4(to_tf32(s2 * vv[0]), to_tf32(s2 * vv[1]), to_tf32(s2 * vv[2]), to_tf32(s2 * vv[3]));
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // ---- dA = [dW | dU] [K1 | V1]^T
  if (tid == 0 && ok) {
    const uint32_t id = idesc_tf32(64, 64);
    const uint32_t r1 = smem_u32(sm + kR1), r2 = smem_u32(sm + kR2), r3 = smem_u32(sm + kR3), r4 = smem_u32(sm + kR4);
    for (int s = 0; s < 16; ++s) mma_tf32_ss(tb + kTdA, desc_kmajor(r3, 8192, s), desc_kmajor(r1, 8192, s), id, s > 0);
    for (int s = 0; s < 16; ++s) mma_tf32_ss(tb + kTdA, desc_kmajor(r4, 8192, s), desc_kmajor(r2, 8192, s), id, true);
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
  // ---- dL = -A^T dA A^T
  uint8_t* sAT = sm + kR3;
  uint8_t* sdAT = sm + kR3 + 16384;
  uint8_t* sA = sm + kR4;
  uint8_t* sX = sm + kR4 + 16384;
  {
    float r[32];
    tmem_ld32(tl + kTdA + 32 * half, r);
    tmem_wait_ld_regs(r);
    if (owner) {
#pragma unroll
      for (int m = 0; m < 32; ++m) put32(sdAT, kC, 32 * half + m, rr, to_tf32(r[m]));
    }
    // A [i][j] read once, coalesced (thread: column j, 16 rows i), into both operands: A^T
    // (row j, four consecutive i per 16-byte chunk) and A (row i, column j)
    const int j = tid & 63, i0 = 16 * (tid >> 6);
    float buf[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) buf[e] = to_tf32(abuf[e]);
#pragma unroll
    for (int e = 0; e < 16; e += 4)
      *reinterpret_cast<float4*>(sAT + sw128_offset(j, i0 + e, kC, 4)) = make_float4(buf[e], buf[e + 1], buf[e + 2], buf[e + 3]);
#pragma unroll
    for (int e = 0; e < 16; ++e) put32(sA, kC, i0 + e, j, buf[e]);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && ok) {
    const uint32_t id = idesc_tf32(64, 64);
    for (int s = 0; s < 8; ++s)
      mma_tf32_ss(tb + kTX, desc_kmajor(smem_u32(sAT), 8192, s), desc_kmajor(smem_u32(sdAT), 8192, s), id, s > 0);
    mma_commit(&bar_mma);
  }
  __syncwarp();
  ok = ok && mbar_wait(&bar_mma, 0, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();
  {
    float r[32];
    tmem_ld32(tl + kTX + 32 * half, r);
    tmem_wait_ld_regs(r);
    if (owner) {
#pragma unroll
      for (int m = 0; m < 32; ++m) put32(sX, kC, rr, 32 * half + m, to_tf32(r[m]));
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && ok) {
    const uint32_t id = idesc_tf32(64, 64);
    for (int s = 0; s < 8; ++s)
      mma_tf32_ss(tb + kTX, desc_kmajor(smem_u32(sX), 8192, s), desc_kmajor(smem_u32(sA), 8192, s), id, s > 0);
    mma_commit(&bar_mma);
  }
  __syncwarp();
  ok = ok && mbar_wait(&bar_mma, 1, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();
  // ---- decayed pair sums on the tensor cores. For i in the 16-row block I (reference row
  // r_I = 16 I) and j <= 16 I + 15, exp(G_ic - G_jc) = P_ic E_I[j][c] with
  // P_ic = exp(G_ic - G_{r_I,c}) <= 1 and E_I[j][c] = exp(G_{r_I,c} - G_jc), which is <= 1 for
  // j < r_I and at most the in-block drop for j in block I (the prepare kernel's factorisation).
  // With D = dL (strictly lower) and N = scale dAqk (lower):
  //   X1_I = P_I (.) D_I (E_I (.) k^),  Y1_I = P_I (.) N_I (E_I (.) k^)     (rows of block I)
  //   Z    = sum_{I >= J(j)} E_I (.) V_I,  V_I[j][c] = sum_{i in I} (D_ij beta_i k^_ic + N_ij q^_ic) P_ic
  // Both products run with the channels on the 128 accumulator lanes (kind::tf32):
  //   round V: V_I^T = XP_I^T MT_I^T, K = the block's 16 rows for D and 16 for N;
  //   round X: [X1 | Y1]_I^T (unscaled) = (E_I (.) k^)^T [D_I ; N_I]^T, K = 16 (I + 1) tokens.
  // The operands: MT [j][k'] and XP^T [c][k'] with k' = 32 I + 16 part + i % 16 (part 0: D and
  // beta k^ P, part 1: N and q^ P); DN [rho][j], rho = k' (the rows D_I, N_I of block I are
  // 32 consecutive rows); EK_I^T [c][j]. Rows past the chunk are zero in D, N, k and q. MT,
  // XP^T and DN are written in one pass; EK^T replaces MT and XP^T once round V is done.
  uint8_t* sMT = sm + kR1;                       // [64][128] tf32, four 8 KB panels (one per block)
  uint8_t* sXP = sm + kR2;                       // [128][128] tf32, four 16 KB panels (R2, R3)
  uint8_t* sDN = sm + kR4;                       // [128][64] tf32, two 16 KB panels
  auto ek_base = [&](int I) -> uint8_t* {        // EK_I^T [128][16 (I + 1)], 16 KB panels, after round V
    return sm + (I == 3 ? kR1 : (I == 2 ? kR2 : (I == 1 ? kR3 : kR3 + 16384)));
  };
  {
    float dl[32], nn[32];
    tmem_ld32(tl + kTX + 32 * half, dl);
    tmem_ld32(tl + kTAqk + 32 * half, nn);
    tmem_wait_ld_regs(dl);
    tmem_wait_ld_regs(nn);
    if (owner) {
      const int i = rr, kq = 32 * (i >> 4) + (i & 15);
      const bool vi = i < len;
#pragma unroll
      for (int j4 = 0; j4 < 32; j4 += 4) {
        float d4[4], n4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 32 * half + j4 + e;
          d4[e] = (j < i && vi) ? to_tf32(-dl[j4 + e]) : 0.f;
          n4[e] = (j <= i && vi) ? to_tf32(scale * nn[j4 + e]) : 0.f;
          put32(sMT, kC, j, kq, d4[e]);
          put32(sMT, kC, j, kq + 16, n4[e]);
        }
        put32x4(sDN, 2 * kC, kq, 32 * half + j4, d4);
        put32x4(sDN, 2 * kC, kq + 16, 32 * half + j4, n4);
      }
    }
  }
  {
    // XP^T: thread (channel cc, blocks 2 half and 2 half + 1), four rows per 16-byte store
    const int c = cc;
#pragma unroll 1
    for (int b = 0; b < 2; ++b) {
      const int I = 2 * half + b, r0 = 16 * I;
      const float gr = sG2[r0 * kP + c];
#pragma unroll
      for (int r4 = 0; r4 < 16; r4 += 4) {
        float xk[4], xq[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = r0 + r4 + e;
          const float P = exp2f(sG2[i * kP + c] - gr);
          xk[e] = to_tf32(s_b[i] * s_rk[i] * bf16_at(sK, i, c) * P);
          xq[e] = to_tf32(s_rq[i] * bf16_at(sQ, i, c) * P);
        }
        put32x4(sXP, kD, c, 32 * I + r4, xk);
        put32x4(sXP, kD, c, 32 * I + 16 + r4, xq);
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && ok) {
    const uint32_t id = idesc_tf32(128, 64), xp = smem_u32(sXP), mt = smem_u32(sMT);
    for (int I = 0; I < 4; ++I)
      for (int s = 0; s < 4; ++s)
        mma_tf32_ss(tb + kTV + 64 * I, desc_kmajor(xp + 16384 * I, 16384, s), desc_kmajor(mt + 8192 * I, 8192, s), id, s > 0);
    mma_commit(&bar_mma);
  }
  __syncwarp();
  ok = ok && mbar_wait(&bar_mma, 0, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();
  __syncthreads();  // MT and XP^T are free: EK^T takes their place
  {
    // EK_I^T rows of token block J for every I >= J: thread (channel cc, blocks {0, 3} or
    // {1, 2}, which balances the halves), four tokens per 16-byte store
    const int c = cc;
#pragma unroll 1
    for (int b = 0; b < 2; ++b) {
      const int J = half == 0 ? 3 * b : 1 + b, r0 = 16 * J;
      const float gJ = sG2[r0 * kP + c];
      float tr[4];
#pragma unroll
      for (int I = 0; I < 4; ++I) tr[I] = I > J ? exp2f(sG2[16 * I * kP + c] - gJ) : 1.f;
#pragma unroll
      for (int r4 = 0; r4 < 16; r4 += 4) {
        float kd[4], x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = r0 + r4 + e;
          kd[e] = s_rk[j] * bf16_at(sK, j, c) * exp2f(gJ - sG2[j * kP + c]);
        }
#pragma unroll
        for (int I = 0; I < 4; ++I) {
          if (I < J) continue;
#pragma unroll
          for (int e = 0; e < 4; ++e) x[e] = to_tf32(tr[I] * kd[e]);
          put32x4(ek_base(I), kD, c, r0 + r4, x);
        }
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && ok) {
    const uint32_t id = idesc_tf32(128, 32), dn = smem_u32(sDN);
    for (int I = 0; I < 4; ++I) {
      const uint32_t ek = smem_u32(ek_base(I));
      for (int s = 0; s < 2 * (I + 1); ++s)
        mma_tf32_ss(tb + kTXY + 32 * I, desc_kmajor(ek, 16384, s), desc_kmajor(dn + 4096 * I, 16384, s), id, s > 0);
    }
    mma_commit(&bar_mma);
  }
  __syncwarp();
  ok = ok && mbar_wait(&bar_mma, 1, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();
  __syncthreads();  // the EK^T operands are free: the accumulators take their places
  // Per (token, channel) results into the dk^ / dq^ / dG accumulators and k^ (.) X1 (dbeta's
  // pair part): thread (channel cc, token blocks {0, 3} or {1, 2}).
  // dG takes each pair through its row (X1, Y1) and its column (Z) with the same tf32 factors
  // that entered the products (recomputed bit for bit: XP for the rows, EK for the columns), so
  // the two sides of every pair cancel exactly over the chunk, as the exact sums do; dk^ and
  // dq^ take the fp32 factors.
  float* sKacc = reinterpret_cast<float*>(sm + kR2);           // dk^ accumulator [64][128]
  float* sQacc = reinterpret_cast<float*>(sm + kR3);           // dq^ accumulator [64][128]
  float* sGacc = reinterpret_cast<float*>(sm + kR4);           // dG accumulator [64][128]
  float* sKX = reinterpret_cast<float*>(sm + kR1);             // k^ (.) X1 [64][128] (DN is dead)
  {
    const int c = cc;
#pragma unroll 1
    for (int b = 0; b < 2; ++b) {
      const int J = half == 0 ? 3 * b : 1 + b, r0 = 16 * J;
      const float gJ = sG2[r0 * kP + c];
      float xy[32], z[16], zg[16], kd[16], ee[16];
      if (ok) {
        tmem_ld32(tl + kTXY + 32 * J, xy);
        tmem_wait_ld_regs(xy);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) xy[e] = 0.f;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const int t = r0 + r;
        ee[r] = exp2f(gJ - sG2[t * kP + c]);
        kd[r] = s_rk[t] * bf16_at(sK, t, c) * ee[r];  // E_J (.) k^, as the operand build has it
        z[r] = 0.f;
        zg[r] = 0.f;
      }
      for (int I = J; I < 4 && ok; ++I) {
        float v[16];
        tmem_ld16(tl + kTV + 64 * I + r0, v);
        tmem_wait_ld_regs(v);
        const float tr = I > J ? exp2f(sG2[16 * I * kP + c] - gJ) : 1.f;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          z[r] = fmaf(tr, v[r], z[r]);
          zg[r] = fmaf(to_tf32(tr * kd[r]), v[r], zg[r]);
        }
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const int t = r0 + r;
        const float g = sG2[t * kP + c];
        const float P = exp2f(g - gJ), E = ee[r];
        const float kb = bf16_at(sK, t, c), qb = bf16_at(sQ, t, c);
        const float kh = s_rk[t] * kb, bt = s_b[t];
        const float x1 = P * xy[r], y1 = P * xy[16 + r];
        const float xk = to_tf32(s_b[t] * s_rk[t] * kb * P), xq = to_tf32(s_rq[t] * qb * P);
        sKacc[t * kD + c] = bt * x1 + E * z[r];
        sQacc[t * kD + c] = y1;
        sGacc[t * kD + c] = xk * xy[r] + xq * xy[16 + r] - zg[r];
        sKX[t * kD + c] = kh * x1;  // dbeta's pair part, summed over the channels by the assembly
      }
    }
  }
  __syncthreads();
  // ---- per-token assembly and L2-norm backward: each warp takes whole token rows, lane l
  // channels 4l .. 4l+3. The row sums over the channels (dbeta, q^ . dq^, k^ . dk^) are one
  // warp reduction each, in a fixed order, and every lane holds them after it, so the row's dq
  // and dk follow at once; each channel's share of dG_last is summed over the warps below.
  const float glc = sG2[(len - 1) * kP + cc];
  {
    const int c4 = 4 * lane;
    const size_t rowbase = tile * kTileW;
    float glc4[4], glp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 4; ++e) glc4[e] = sG2[(len - 1) * kP + c4 + e];
    for (int t = warp; t < len; t += kThreads / 32) {
      const size_t o = rowbase + size_t(t) * kD + c4;
      const float4 dqt4 = ldg_bf16x4(p.dQt + o);
      const float4 dk14 = ldg_bf16x4(p.dK1 + o);
      const float4 dkt4 = ldg_bf16x4(p.dKt + o);
      const float4 dv14 = __ldg(reinterpret_cast<const float4*>(p.dV1 + o));
      const float dqt[4] = {dqt4.x, dqt4.y, dqt4.z, dqt4.w}, dk1[4] = {dk14.x, dk14.y, dk14.z, dk14.w};
      const float dkt[4] = {dkt4.x, dkt4.y, dkt4.z, dkt4.w}, dv1[4] = {dv14.x, dv14.y, dv14.z, dv14.w};
      float qv[4], kv[4], vv[4];
      bf16x4_at(sQ, t, c4, qv);
      bf16x4_at(sK, t, c4, kv);
      bf16x4_at(sV, t, c4, vv);
      const float rq = s_rq[t], rk = s_rk[t], bt = s_b[t];
      const float4 qa = *reinterpret_cast<const float4*>(sQacc + t * kD + c4);
      const float4 ka = *reinterpret_cast<const float4*>(sKacc + t * kD + c4);
      float4* ga4 = reinterpret_cast<float4*>(sGacc + t * kD + c4);
      const float4 ga = *ga4;
      float qacc[4] = {qa.x, qa.y, qa.z, qa.w}, kacc[4] = {ka.x, ka.y, ka.z, ka.w}, gacc[4] = {ga.x, ga.y, ga.z, ga.w};
      const float4 kx = *reinterpret_cast<const float4*>(sKX + t * kD + c4);
      float sdb = (kx.x + kx.y) + (kx.z + kx.w), sq = 0.f, sk = 0.f, dvo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float G = sG2[t * kP + c4 + e];
        const float eG = exp2f(G), eL = exp2f(glc4[e] - G);
        const float qh = rq * qv[e], kh = rk * kv[e];
        const float dqh = qacc[e] + scale * eG * dqt[e];
        const float dkh = kacc[e] + bt * eG * dk1[e] + eL * dkt[e];
        qacc[e] = dqh;
        kacc[e] = dkh;
        gacc[e] += bt * eG * dk1[e] * kh + scale * eG * dqt[e] * qh - eL * dkt[e] * kh;
        glp[e] = fmaf(eL * dkt[e], kh, glp[e]);
        dvo[e] = bt * dv1[e];
        sdb += eG * dk1[e] * kh + dv1[e] * vv[e];
        sq += dqh * qh;
        sk += dkh * kh;
      }
      *ga4 = make_float4(gacc[0], gacc[1], gacc[2], gacc[3]);
      *reinterpret_cast<uint2*>(p.dv + (size_t(ch.x + t) * H + h) * kD + c4) = pack_bf16x4(dvo);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        sdb += __shfl_xor_sync(0xffffffffu, sdb, off);
        sq += __shfl_xor_sync(0xffffffffu, sq, off);
        sk += __shfl_xor_sync(0xffffffffu, sk, off);
      }
      if (lane == 0) s_dba[0][t] = sdb;
      float dq[4], dk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        dq[e] = p.l2norm ? rq * (qacc[e] - rq * qv[e] * sq) : qacc[e];
        dk[e] = p.l2norm ? rk * (kacc[e] - rk * kv[e] * sk) : kacc[e];
      }
      if (p.dq32) {  // per value head, summed over the q/k group later
        const size_t oq = (size_t(ch.x + t) * H + h) * kD + c4;
        *reinterpret_cast<float4*>(p.dq32 + oq) = make_float4(dq[0], dq[1], dq[2], dq[3]);
        *reinterpret_cast<float4*>(p.dk32 + oq) = make_float4(dk[0], dk[1], dk[2], dk[3]);
      } else {
        const size_t oq = (size_t(ch.x + t) * (H / p.qk_group) + h) * kD + c4;
        *reinterpret_cast<uint2*>(p.dq + oq) = pack_bf16x4(dq);
        *reinterpret_cast<uint2*>(p.dk + oq) = pack_bf16x4(dk);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) s_glw[warp][c4 + e] = glp[e];
  }
  __syncthreads();
  // ---- dg by reverse cumulative sum per channel
  if (half == 0) {
    float acc = exp2f(glc) * dgam_c;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) acc += s_glw[w][cc];   // dG_last shares, in warp order
    if (p.gate_act) {
      // chain rule through the safe gate g = lb sigmoid(z), z = a (x + dt_bias), a = exp(A_log):
      // dx = dg lb s (1 - s) a; the parameter gradients are summed per chunk here and over the
      // chunks by the gate-gradient kernel
      const float a = expf(p.A_log[h]), dtb = p.dt_bias[h * kD + cc];
      float pa = 0.f, pd = 0.f;
      for (int t = len - 1; t >= 0; --t) {
        acc += sGacc[t * kD + cc];
        const size_t o = (size_t(ch.x + t) * H + h) * kD + cc;
        const float z = a * (p.g[o] + dtb);
        const float sg = 1.f / (1.f + expf(-z));
        const float dsz = acc * p.lower_bound * sg * (1.f - sg);
        const float dx = dsz * a;
        p.dg[o] = dx;
        pa = fmaf(dsz, z, pa);
        pd += dx;
      }
      p.dA_part[tile * kD + cc] = pa;
      p.ddt_part[tile * kD + cc] = pd;
    } else {
      for (int t = len - 1; t >= 0; --t) {
        acc += sGacc[t * kD + cc];
        p.dg[(size_t(ch.x + t) * H + h) * kD + cc] = acc;
      }
    }
  }
  if (tid < len) {
    float db = s_dba[0][tid];
    if (p.beta_sigmoid) db *= s_b[tid] * (1.f - s_b[tid]);
    p.dbeta[size_t(ch.x + tid) * H + h] = __float2bfloat16_rn(db);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 512);
}

cudaError_t launch_bwd_tok_kda(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                               const CUtensorMap& mVN, const CUtensorMap& mDW, const CUtensorMap& mDVN,
                               const CUtensorMap& mdO, const BwdTokParams& p, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_bwd_tok_kda, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(unsigned(p.NC) * unsigned(p.hgn));
  k_bwd_tok_kda<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, mVN, mDW, mDVN, mdO, p);
  return cudaGetLastError();
}

}  // namespace gdn
