// Prepare kernel (Gated DeltaNet, scalar gate): everything of a chunk that does not depend
// on the carried state, for two chunks per CTA.
//
// Per chunk (the eager reference `torch_chunk_gated_delta_rule`, hyper-parallel GDN Diff
// Coverage page, steps before its chunk loop):
//   r_q, r_k   = rsqrt(|q|^2 + 1e-6), rsqrt(|k|^2 + 1e-6)            (`_l2norm`)
//   G          = chunk-local cumulative gate                          (`g.cumsum(-1)`)
//   L_ij       = beta_i r_i r_j (k_i . k_j) exp(G_i - G_j), i > j     (`attn`, strictly lower)
//   A          = (I + L)^-1                                           (row loop + identity)
//   W          = A diag(beta exp(G) r_k) k                            (`k_cumdecay`)
//   U          = A diag(beta) v                                       (`value`)
//   Aqk_ij     = scale r_q,i r_k,j (q_i . k_j) exp(G_i - G_j), i >= j (chunk-loop `attn`)
//   Qt         = scale r_q exp(G) q ;  KtT = (r_k exp(G_last - G) k)^T ; gam = exp(G_last)
//
// GB300 mapping. The two chunks of a CTA are stacked into one 128-row tile so every
// tensor-core product is a 128-lane tcgen05 MMA: the Gram products K K^T and Q K^T
// (raw bf16 tiles straight from TMA, so the operands are exact) land in TMEM and only their
// two diagonal 64x64 blocks are used; W and U are block-diagonal (A) times the raw k / v tile
// (MN-major B operand). L2-norm factors and decays are applied to the fp32 MMA results, never
// to the bf16 operands. Eight warps share the work: two threads per row of the stacked tile
// (TMEM lane = row), each covering half of its columns. The unit-lower-triangular inverse runs
// in fp32 registers, one column per lane pair (forward substitution, the same recurrence as
// the page's row loop). Row-major
// output tiles (Qt, Kt, Aqk, W, U) are staged in shared memory in the swizzled operand layout
// and written by TMA stores, so the row-per-thread results leave as whole lines; the
// transposed tiles are written directly (consecutive threads, consecutive addresses).
#include "common.cuh"
#include "tri_inverse.cuh"
#include "umma.cuh"

namespace gdn {

namespace {

constexpr int kThreads = 256;  // two threads per row of the stacked 128-row tile
constexpr int kRows = 128;
constexpr uint32_t kPanel = 16384;  // 128 rows x 128 B
constexpr uint32_t kOffQ = 0, kOffK = 32768, kOffV = 65536, kOffA1 = 98304, kOffA2 = 131072,
                   kOffL = 163840, kOffS0 = 196608, kSmemBytes = 229376 + 1024;
constexpr uint32_t kStage = 32768;  // one chunk's [64][128] fp32 tile: 4 panels x 64 rows x 128 B

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 t = __bfloat1622float2(b[e]);
    f[2 * e] = t.x;
    f[2 * e + 1] = t.y;
  }
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    k_prep_gdn(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mQt,
               const __grid_constant__ CUtensorMap mKt, const __grid_constant__ CUtensorMap mAqk,
               const __grid_constant__ CUtensorMap mW, const __grid_constant__ CUtensorMap mU, const PrepParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1k(smem_raw);
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sK = sm + kOffK;
  uint8_t* sV = sm + kOffV;
  uint8_t* sA1 = sm + kOffA1;
  uint8_t* sA2 = sm + kOffA2;
  float* sL = reinterpret_cast<float*>(sm + kOffL);
  uint8_t* sS0 = sm + kOffS0;
  __shared__ uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;
  __shared__ float s_g[kRows], s_rk[kRows], s_G2[kRows];  // s_G2 = G log2(e)
  __shared__ int4 s_chunk[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // heads fastest: the CTAs in flight share token rows of q, k, v and neighbouring tiles
  const int h = int(blockIdx.x % p.hgn) + p.hg0, pair = int(blockIdx.x / p.hgn), H = p.H;
  // Row of the stacked tile (= TMEM lane) and column half of this thread.
  const int rt = tid & (kRows - 1), hf = tid >> 7;
  const int blk = rt >> 6, il = rt & 63;

  if (warp == 0) tmem_alloc(&tslot, 256);
  if (tid == 0) {
    // the barriers are this thread's alone until the block barrier below: start the loads now
    int4 cb[2];
    for (int b = 0; b < 2; ++b) cb[b] = 2 * pair + b < p.NC ? chunk_entry(p.chunks, 2 * pair + b, p.dense_T) : make_int4(0, 0, 0, 0);
    abort_flag = 0;
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    const int nexist = (cb[0].y > 0) + (cb[1].y > 0);
    mbar_expect_tx(&bar_tma, uint32_t(nexist) * 6u * 8192u);
    for (int b = 0; b < 2; ++b) {
      s_chunk[b] = cb[b];
      if (cb[b].y <= 0) continue;
      for (int pp = 0; pp < 2; ++pp) {
        const int x = h * kD + 64 * pp, xqk = (h / p.qk_group) * kD + 64 * pp, y = cb[b].x;
        tma_load_2d(sQ + pp * kPanel + b * 8192, &mq, xqk, y, &bar_tma);
        tma_load_2d(sK + pp * kPanel + b * 8192, &mk, xqk, y, &bar_tma);
        tma_load_2d(sV + pp * kPanel + b * 8192, &mv, x, y, &bar_tma);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  const uint32_t lane_base = tmem_lane_base(warp);
  const int4 ch = s_chunk[blk];
  const int len = ch.y;
  const int c_idx = 2 * pair + blk;
  const bool valid = il < len;
  const int row = ch.x + il;

  // A missing second chunk leaves its tile rows unloaded: zero them so that the products
  // with zero coefficients stay exactly zero.
  if (len == 0) {
#pragma unroll
    for (int c16 = 8 * hf; c16 < 8 * hf + 8; ++c16) {
      const uint32_t off = sw128_offset(rt, c16 * 8, 128, 2);
      *reinterpret_cast<uint4*>(sQ + off) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sK + off) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sV + off) = make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();
  }
  float gi = 0.f, bi = 0.f;
  if (valid) {
    gi = fmaxf(p.g[size_t(row) * H + h], kGateFloor);  // g = -inf: exact reset, finite cumsum
    bi = __bfloat162float(p.beta[size_t(row) * H + h]);
    if (p.beta_sigmoid) bi = 1.f / (1.f + expf(-bi));
  }
  if (hf == 0) {
    s_g[rt] = gi;
  }
  mbar_wait(&bar_tma, 0, &abort_flag, p.status, kDevTimeoutTma);

  // L2-norm factors from the staged rows: each half-row's partial sums meet in the A1 area,
  // which is free until Qt is staged there.
  {
    float ssq = 0.f, ssk = 0.f;
#pragma unroll
    for (int c16 = 8 * hf; c16 < 8 * hf + 8; ++c16) {
      const uint32_t off = sw128_offset(rt, c16 * 8, 128, 2);
      float f[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(sQ + off), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) ssq = fmaf(f[e], f[e], ssq);
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(sK + off), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) ssk = fmaf(f[e], f[e], ssk);
    }
    float* part = reinterpret_cast<float*>(sA1);
    part[tid] = ssq;
    part[kThreads + tid] = ssk;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Gram products: TMEM cols [0,128) = K K^T, [128,256) = Q K^T (pair-stacked). They read only
  // the raw tiles, so they start here, under the norms and the gate cumsum.
  if (tid == 0 && !abort_flag) {
    const uint32_t id = idesc_bf16(128, 128);
    const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK);
    for (int s = 0; s < 8; ++s) mma_bf16_ss(tb, desc_kmajor(k0, kPanel, s), desc_kmajor(k0, kPanel, s), id, s > 0);
    for (int s = 0; s < 8; ++s)
      mma_bf16_ss(tb + 128, desc_kmajor(q0, kPanel, s), desc_kmajor(k0, kPanel, s), id, s > 0);
    mma_commit(&bar_mma);
  }
  const float* part = reinterpret_cast<const float*>(sA1);
  const float rq = p.l2norm ? 1.f / sqrtf(part[rt] + part[rt + kRows] + 1e-6f) : 1.f;
  const float rk = p.l2norm ? 1.f / sqrtf(part[kThreads + rt] + part[kThreads + rt + kRows] + 1e-6f) : 1.f;
  // G = chunk-local cumulative gate of row il: an inclusive scan over the warp's 32 rows plus,
  // for rows 32..63, the total of rows 0..31 (a warp sum)
  float G = s_g[rt];
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, G, off);
    if (lane >= off) G += y;
  }
  if (il >= 32) {
    float base = s_g[blk * kC + lane];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) base += __shfl_xor_sync(0xffffffffu, base, off);
    G += base;
  }
  if (hf == 0) {
    s_rk[rt] = rk;
    s_G2[rt] = G * kLog2e;  // exp(G_i - G_j) = exp2(G2_i - G2_j)
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const float Glast2 = len > 0 ? s_G2[blk * kC + len - 1] : 0.f;  // G_last log2(e)


  // Gated queries and end-decayed keys (state-independent operands of the chunk loop): the
  // row-major Qt and Kt tiles are staged (A1/A2 and L/S0 are free until the inverse) and
  // stored by TMA; the transposed KtT and QtT go straight out. Each thread covers half a row.
  const size_t tile = size_t(c_idx) * H + h;
  uint8_t* stQt = blk ? sA2 : sA1;
  uint8_t* stKt = blk ? sS0 : reinterpret_cast<uint8_t*>(sL);
  if (len > 0) {
    const float fq = valid ? p.scale * rq * expf(G) : 0.f;
    const float fk = valid ? rk * exp2f(Glast2 - G * kLog2e) : 0.f;
    float* ktt = p.KtT + tile * kTileKtT + il;
#pragma unroll
    for (int c16 = 8 * hf; c16 < 8 * hf + 8; ++c16) {
      const uint32_t off = sw128_offset(rt, c16 * 8, 128, 2);
      float f[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(sQ + off), f);
#pragma unroll
      for (int e = 0; e < 8; e += 4)
        *reinterpret_cast<float4*>(stQt + sw128_offset(il, c16 * 8 + e, kC, 4)) =
            make_float4(to_tf32(f[e] * fq), to_tf32(f[e + 1] * fq), to_tf32(f[e + 2] * fq), to_tf32(f[e + 3] * fq));
      if (p.QtT) {
#pragma unroll
        for (int e = 0; e < 8; ++e) p.QtT[tile * kTileKtT + size_t(c16 * 8 + e) * kC + il] = to_tf32(f[e] * fq);
      }
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(sK + off), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) ktt[size_t(c16 * 8 + e) * kC] = to_tf32(f[e] * fk);
      if (p.Kt) {
#pragma unroll
        for (int e = 0; e < 8; e += 4)
          *reinterpret_cast<float4*>(stKt + sw128_offset(il, c16 * 8 + e, kC, 4)) =
              make_float4(to_tf32(f[e] * fk), to_tf32(f[e + 1] * fk), to_tf32(f[e + 2] * fk), to_tf32(f[e + 3] * fk));
      }
    }
    if (hf == 0) {
      if (il == 0) p.gam[tile * kD] = exp2f(Glast2);
      if (p.Gc) p.Gc[tile * kC + il] = G;
      if (p.rq) p.rq[tile * kC + il] = rq;
      if (p.rk) p.rk[tile * kC + il] = rk;
      if (p.beff) p.beff[tile * kC + il] = bi;
    }
  }
  fence_async_smem();
  __syncthreads();
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      if (s_chunk[b].y <= 0) continue;
      const int y = (int(2 * pair + b) * H + h) * kC;
      for (int pp = 0; pp < 4; ++pp) {
        tma_store_2d(&mQt, pp * 32, y, (b ? sA2 : sA1) + pp * 8192);
        if (p.Kt) tma_store_2d(&mKt, pp * 32, y, (b ? sS0 : reinterpret_cast<uint8_t*>(sL)) + pp * 8192);
      }
    }
    tma_store_commit();
  }
  const bool ok1 = mbar_wait(&bar_mma, 0, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();
  if (tid == 0) tma_store_wait_read();  // L and A1 are rewritten next
  __syncthreads();
  uint8_t* stAqk = sA1 + blk * (kStage / 2);
  if (ok1) {
    // this thread's 32 columns j = 32 hf + jj of the chunk's 64x64 blocks
    float* LT = sL + blk * (kC * kC) + il;  // column il of L^T
    float kk[32], qk[32];
    tmem_ld32(tb + lane_base + blk * kC + 32 * hf, kk);
    tmem_ld32(tb + lane_base + 128 + blk * kC + 32 * hf, qk);
    tmem_wait_ld_regs(kk);
    tmem_wait_ld_regs(qk);
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const int j = 32 * hf + jj, pj = blk * kC + j;
      const float dec = exp2f(G * kLog2e - s_G2[pj]) * s_rk[pj];
      LT[j * kC] = (j < il) ? bi * rk * kk[jj] * dec : 0.f;
      qk[jj] = (j <= il && valid) ? to_tf32(p.scale * rq * qk[jj] * dec) : 0.f;
    }
    if (len > 0) {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        *reinterpret_cast<float4*>(stAqk + sw128_offset(il, 32 * hf + 4 * e, kC, 4)) =
            make_float4(qk[4 * e], qk[4 * e + 1], qk[4 * e + 2], qk[4 * e + 3]);
      if (p.AqkT) {
        float* at = p.AqkT + tile * kTileAqk + il;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) at[size_t(32 * hf + jj) * kC] = qk[jj];
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      if (s_chunk[b].y <= 0) continue;
      const int y = (int(2 * pair + b) * H + h) * kC;
      for (int pp = 0; pp < 2; ++pp) tma_store_2d(&mAqk, pp * 32, y, sA1 + b * (kStage / 2) + pp * 8192);
    }
    tma_store_commit();
  }

  // A = (I + L)^-1 per chunk, one column per lane pair (into sX, which reuses the q tile: q is
  // no longer needed once Qt and the Q K^T product are done); then the scaled block-diagonal
  // operands A1 = A diag(beta exp(G) r_k) and A2 = A diag(beta), bf16, K-major, 128x128, with
  // the unit diagonal left out (added in fp32 after the MMA).
  {
    // The columns of the first 16-row block cost the most; the second chunk takes its blocks in
    // reverse so that warps w and w + 4 (one SM sub-partition) share the work evenly.
    const int cb = warp >> 2, cc = 16 * (cb ? 3 - (warp & 3) : (warp & 3)) + (lane & 15);
    unit_lower_inverse_column(sL + cb * (kC * kC), reinterpret_cast<float*>(sQ) + cb * (kC * kC), cc, lane >> 4);
  }
  if (tid == 0) tma_store_wait_read();  // A1 held the staged Aqk tiles
  __syncthreads();
  const float* sX = reinterpret_cast<const float*>(sQ) + blk * (kC * kC);
  if (p.A && len > 0) {
    float* a = p.A + tile * kTileAqk + il;
    for (int r = 32 * hf; r < 32 * hf + 32; ++r) a[size_t(r) * kC] = sX[r * kC + il];
  }
  {
    const float s1 = bi * expf(G) * rk, s2 = bi;
    const int col = rt;
    const __nv_bfloat16 z = __float2bfloat16_rn(0.f);
    const int other = (blk ^ 1) * kC;
#pragma unroll 4
    for (int r = 32 * hf; r < 32 * hf + 32; ++r) {
      const float xr = r == il ? 0.f : sX[r * kC + il];
      const uint32_t own = sw128_offset(blk * kC + r, col, 128, 2);
      *reinterpret_cast<__nv_bfloat16*>(sA1 + own) = __float2bfloat16_rn(xr * s1);
      *reinterpret_cast<__nv_bfloat16*>(sA2 + own) = __float2bfloat16_rn(xr * s2);
      const uint32_t off = sw128_offset(other + r, col, 128, 2);
      *reinterpret_cast<__nv_bfloat16*>(sA1 + off) = z;
      *reinterpret_cast<__nv_bfloat16*>(sA2 + off) = z;
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // W = A1 k (TMEM cols [0,128)), U = A2 v (cols [128,256)); k, v as MN-major B operands.
  // A1, A2 carry only the strictly lower part of A (bf16); the identity part, which dominates
  // W and U, is added in fp32 from the exact inputs: W_i += beta_i exp(G_i) r_i k_i,
  // U_i += beta_i v_i. This keeps the bf16 rounding confined to the small off-diagonal terms.
  if (tid == 0 && !abort_flag) {
    const uint32_t id = idesc_bf16(128, 128, false, true);
    const uint32_t a1 = smem_u32(sA1), a2 = smem_u32(sA2), k0 = smem_u32(sK), v0 = smem_u32(sV);
    for (int s = 0; s < 8; ++s) mma_bf16_ss(tb, desc_kmajor(a1, kPanel, s), desc_mnmajor_bf16(k0, kPanel, s), id, s > 0);
    for (int s = 0; s < 8; ++s)
      mma_bf16_ss(tb + 128, desc_kmajor(a2, kPanel, s), desc_mnmajor_bf16(v0, kPanel, s), id, s > 0);
    mma_commit(&bar_mma);
  }
  const bool ok2 = mbar_wait(&bar_mma, 1, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();
  // Warps 0-3 finish W (staged in L for chunk 0, S0 for chunk 1), warps 4-7 finish U (staged
  // in A1 / A2, free once the MMAs are done).
  if (ok2 && len > 0) {
    const int which = hf;
    const float sc = which == 0 ? bi * expf(G) * rk : bi;
    uint8_t* stage = which == 0 ? (blk ? sS0 : reinterpret_cast<uint8_t*>(sL)) : (blk ? sA2 : sA1);
    const uint8_t* src = which == 0 ? sK : sV;
    for (int half = 0; half < 2; ++half) {
      float r[64];
      tmem_ld64(tb + lane_base + which * 128 + half * 64, r);
      tmem_wait_ld_regs(r);
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        float in[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(src + sw128_offset(rt, half * 64 + c8 * 8, 128, 2)), in);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float val = fmaf(sc, in[e], r[c8 * 8 + e]);
          r[c8 * 8 + e] = which == 0 ? to_tf32(val) : val;
        }
      }
#pragma unroll
      for (int e = 0; e < 16; ++e)
        *reinterpret_cast<float4*>(stage + sw128_offset(il, half * 64 + 4 * e, kC, 4)) =
            make_float4(r[4 * e], r[4 * e + 1], r[4 * e + 2], r[4 * e + 3]);
      if (which == 0 && p.WT) {
        float* wt = p.WT + tile * kTileKtT + size_t(half * 64) * kC + il;
#pragma unroll
        for (int e = 0; e < 64; ++e) wt[size_t(e) * kC] = r[e];
      }
    }
  }
  fence_async_smem();
  __syncthreads();
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      if (s_chunk[b].y <= 0 || !ok2) continue;
      const int y = (int(2 * pair + b) * H + h) * kC;
      for (int pp = 0; pp < 4; ++pp) {
        tma_store_2d(&mW, pp * 32, y, (b ? sS0 : reinterpret_cast<uint8_t*>(sL)) + pp * 8192);
        tma_store_2d(&mU, pp * 32, y, (b ? sA2 : sA1) + pp * 8192);
      }
    }
    tma_store_commit();
    tma_store_wait_read();  // the writes themselves complete before the grid does
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 256);
}

cudaError_t launch_prep_gdn(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const CUtensorMap& mQt, const CUtensorMap& mKt, const CUtensorMap& mAqk,
                            const CUtensorMap& mW, const CUtensorMap& mU, const PrepParams& p, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_prep_gdn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(unsigned((p.NC + 1) / 2) * unsigned(p.hgn));
  k_prep_gdn<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, mQt, mKt, mAqk, mW, mU, p);
  return cudaGetLastError();
}

}  // namespace gdn
