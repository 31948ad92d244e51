// Prepare kernel for Kimi Delta Attention (per-channel gate), one chunk per CTA of eight warps.
//
// With G[t][c] the chunk-local cumulative gate of key channel c (the `gk` slot of the KDA
// staged native interface, `_KDAPrepared.gk`, kimi_delta_attention_ascendc.py coverage page)
// and k^, q^ the L2-normalised rows, the chunk quantities are those of the scalar-gate
// prepare kernel with every decay taken per channel:
//   L_ij   = beta_i sum_c k^_ic k^_jc exp(G_ic - G_jc), i > j;      A = (I + L)^-1
//   Aqk_ij = scale sum_c q^_ic k^_jc exp(G_ic - G_jc), i >= j
//   W      = A K1,  K1_jc = beta_j exp(G_jc) k^_jc;                 U = A diag(beta) v
//   Qt_ic  = scale exp(G_ic) q^_ic;  KtT_ci = exp(G_last,c - G_ic) k^_ic;  gam_c = exp(G_last,c)
//
// GB300 mapping. exp(G_ic - G_jc) does not factor into bounded row and column terms over a
// whole chunk (G spans tens of units), so each 16-row block I of the chunk gets its own
// reference row r_I = 16 I: exp(G_ic - G_jc) = exp(G_ic - G_{r_I,c}) exp(G_{r_I,c} - G_jc).
// For i in block I the first factor is <= 1, and for j < r_I the second one is too; for j in
// block I it is at most the decay across 15 tokens. One stacked 128-row tf32 operand (keys
// then queries, each row scaled by its block's reference) times B_I = k^ exp(G_{r_I} - G)
// (rows j <= 16 I + 15, so N = 16 (I + 1)) gives, in four 128-lane MMAs, every row block of
// both L and Aqk. Row j of B_I splits again at j's own block J: exp(G_{r_I} - G_j) =
// exp(G_{r_I} - G_{r_J}) exp(G_{r_J} - G_j), a per-channel factor of the block pair (<= 1 for
// J < I) times the reciprocal of the stacked operand's factor of row j, so each element of the
// chunk takes two exponentials for all five operands.
// The unit-lower inverse and the WY products follow the scalar-gate kernel: W's right factor
// carries the per-channel decay (tf32, thread-written); U uses the raw v tile (bf16); the
// unit diagonal of A is applied in fp32 from the exact inputs. Exponentials that only feed
// tf32-rounded operands use the hardware exponential (__expf: a few fp32 ulps, far inside the
// 2^-11 of tf32); gam, an fp32 output of the state chain, keeps expf.
#include "common.cuh"
#include "tri_inverse.cuh"
#include "umma.cuh"

namespace gdn {

namespace {

constexpr int kThreads = 256;  // eight warps: two threads per row or channel in most phases
constexpr int kGP = kD + 1;                                // padded row stride of G (floats)
constexpr uint32_t kOffQ = 0, kOffK = 16384, kOffV = 32768;  // bf16 [64][128] tiles
constexpr uint32_t kOffG = 49152;                          // fp32 [64][129]
constexpr uint32_t kOffAS = 83968;                         // stacked A operand, tf32 [128][128] (64 KB)
constexpr uint32_t kOffB = 149504;                         // B_3, B_2, B_0: tf32 [64 / 48 / 16][128]
constexpr uint32_t kSmemBytes = kOffB + 65536 + 1024;
// B_I (N = 16 (I + 1) rows) offsets; B_1 borrows the value tile's slot, whose load is issued once
// the Gram products are done.
__device__ __forceinline__ uint32_t b_off(int I) {
  return I == 3 ? kOffB : (I == 2 ? kOffB + 32768 : (I == 1 ? kOffV : kOffB + 57344));
}
// Later phases reuse the operand region [kOffAS, kOffB + 64 KB):
constexpr uint32_t kOffLT = kOffAS;                        // L^T fp32 [64][64]
constexpr uint32_t kOffX = kOffAS + 16384;                 // inverse columns fp32 [64][64]
constexpr uint32_t kOffA1 = kOffAS + 32768;                // (A - I) diag(beta r_k), tf32 [64][64]
constexpr uint32_t kOffA2 = kOffAS + 49152;                // (A - I) diag(beta), bf16 [64][64]
constexpr uint32_t kOffK1T = kOffB;                        // (k (.) exp(G))^T, tf32 [128][64]
constexpr int kAP = kC + 1;                                // padded row stride of the Aqk staging
constexpr uint32_t kOffAqkS = kOffB + 32768;               // Aqk staging fp32 [64][65] (beside K1T)
static_assert(kOffAqkS + 4 * kC * kAP <= kOffB + 65536, "Aqk staging fits the B region");

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}
__device__ __forceinline__ float bf16_at(const uint8_t* tile, int row, int col) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + sw128_offset(row, col, kC, 2)));
}
__device__ __forceinline__ void put32(uint8_t* tile, int rows, int row, int col, float x) {
  *reinterpret_cast<float*>(tile + sw128_offset(row, col, rows, 4)) = x;
}
__device__ __forceinline__ void put_tf32x8(uint8_t* tile, int rows, int row, int col, const float* f) {
  *reinterpret_cast<float4*>(tile + sw128_offset(row, col, rows, 4)) = make_float4(f[0], f[1], f[2], f[3]);
  *reinterpret_cast<float4*>(tile + sw128_offset(row, col + 4, rows, 4)) = make_float4(f[4], f[5], f[6], f[7]);
}
__device__ __forceinline__ void st_f32x8(float* dst, const float* f) {
  reinterpret_cast<float4*>(dst)[0] = make_float4(f[0], f[1], f[2], f[3]);
  reinterpret_cast<float4*>(dst)[1] = make_float4(f[4], f[5], f[6], f[7]);
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
    k_prep_kda(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const PrepParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1k(smem_raw);
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sK = sm + kOffK;
  uint8_t* sV = sm + kOffV;
  float* sG = reinterpret_cast<float*>(sm + kOffG);
  __shared__ uint64_t bar_tma, bar_v, bar_mma;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;
  __shared__ float s_rq[kC], s_rk[kC], s_b[kC], s_gl[kD];
  __shared__ __align__(16) float s_T[6][kD];  // exp(G_{r_I} - G_{r_J}), J < I, at I (I - 1) / 2 + J

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hf = tid >> 7;     // which half of the block (rows or columns, per phase)
  // heads fastest: the CTAs in flight share token rows of the inputs and neighbouring tiles
  const int c_idx = int(blockIdx.x / p.hgn), h = int(blockIdx.x % p.hgn) + p.hg0, H = p.H;
  const size_t tile = size_t(c_idx) * H + h;
  const ChunkEntry ch = chunk_entry(p.chunks, c_idx, p.dense_T);
  const int len = ch.y;

  if (warp == 0) tmem_alloc(&tslot, 256);
  if (tid == 0) {
    // the barriers are this thread's alone until the block barrier below: start the loads now
    abort_flag = 0;
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_v, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    mbar_expect_tx(&bar_tma, 2u * 16384u);
    for (int pp = 0; pp < 2; ++pp) {
      const int xqk = (h / p.qk_group) * kD + 64 * pp;
      tma_load_2d(sQ + pp * 8192, &mq, xqk, ch.x, &bar_tma);
      tma_load_2d(sK + pp * 8192, &mk, xqk, ch.x, &bar_tma);
    }
  }
  // Cumulative gate of channel c: each half sums its 32 rows; the second half adds the first
  // half's total after the barrier (rows past the chunk repeat the last value).
  {
    const int c = tid & 127, t0 = 32 * hf;
    const float* src = p.g + (size_t(ch.x) * H + h) * kD + c;
    float buf[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) buf[e] = (t0 + e < len) ? src[size_t(t0 + e) * H * kD] : 0.f;
    if (p.gate_act) {
      // safe gate from the logits: lower_bound * sigmoid(exp(A_log) (x + dt_bias))
      const float a = expf(p.A_log[h]), dtb = p.dt_bias[h * kD + c];
#pragma unroll
      for (int e = 0; e < 32; ++e)
        buf[e] = (t0 + e < len) ? p.lower_bound / (1.f + expf(-a * (buf[e] + dtb))) : 0.f;
    }
    float run = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      run += buf[e];
      sG[(t0 + e) * kGP + c] = run;
    }
  }
  if (tid < kC) {
    float b = 0.f;
    if (tid < len) {
      b = __bfloat162float(p.beta[size_t(ch.x + tid) * H + h]);
      if (p.beta_sigmoid) b = 1.f / (1.f + expf(-b));
    }
    s_b[tid] = b;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (hf == 1) {
    const int c = tid & 127;
    const float base = sG[31 * kGP + c];
#pragma unroll 8
    for (int t = 32; t < kC; ++t) sG[t * kGP + c] += base;
  }
  const uint32_t tb = tslot;
  const uint32_t tl = tb + tmem_lane_base(warp);
  mbar_wait(&bar_tma, 0, &abort_flag, p.status, kDevTimeoutTma);
  // rows past the chunk belong to the next document (or are zero): clear them
  if (tid >= len && tid < kC) {
    for (int c16 = 0; c16 < 16; ++c16) {
      const uint32_t off = sw128_offset(tid, c16 * 8, kC, 2);
      *reinterpret_cast<uint4*>(sQ + off) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sK + off) = make_uint4(0, 0, 0, 0);
    }
  }
  __syncthreads();
  // Domain of the block factorisation below: within each 16-row block the cumulative gate of
  // every channel stays within kKdaBlockDropMax of its value at the block's first row (NaN and
  // infinite gates fail the test too). Outside it the results are not defined and the status
  // word reports kDevGateRange.
  {
    const int c = tid & 127;
    bool bad = false;  // accumulated without short-circuiting, so the loads all go out at once
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int r = 16 * (2 * hf + b);
      const float gr = sG[r * kGP + c];
#pragma unroll
      for (int e = 1; e < 16; ++e)
        bad |= (r + e < len) & !(fabsf(sG[(r + e) * kGP + c] - gr) <= kKdaBlockDropMax);
    }
    if (bad && p.status) atomicCAS(p.status, 0, kDevGateRange);
    for (int pr = hf; pr < 6; pr += 2) {
      const int I = pr == 0 ? 1 : (pr < 3 ? 2 : 3), J = pr - I * (I - 1) / 2;
      s_T[pr][c] = __expf(sG[16 * I * kGP + c] - sG[16 * J * kGP + c]);
    }
  }
  // L2-norm factors: thread pairs (2 p, 2 p + 1) share row p % 64 of q (p < 64) or k, half the
  // columns each (eight per load).
  {
    const int pr = tid >> 1, part = tid & 1, t = pr & 63;
    const uint8_t* src = pr < kC ? sQ : sK;
    float ss = 0.f;
#pragma unroll
    for (int c16 = 8 * part; c16 < 8 * part + 8; ++c16) {
      float f[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(src + sw128_offset(t, c16 * 8, kC, 2)), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    const float r = p.l2norm ? 1.f / sqrtf(ss + 1e-6f) : 1.f;
    if (part == 0) {
      if (pr < kC) s_rq[t] = r; else s_rk[t] = r;
    }
  }
  if (tid < kD) s_gl[tid] = sG[(len - 1) * kGP + tid];
  __syncthreads();

  // One pass builds the stacked operand (rows 0..63 k^_j P_j, rows 64..127 q^_j P_j, with
  // P_j = exp(G_j - G_{r(j)}) <= 1) and every B_I row of token j: k^_j / P_j for I = J, times
  // exp(G_{r_I} - G_{r_J}) for I > J. Warp w takes the 16 tokens of block J (w < 4: J = w;
  // otherwise J = 7 - w, so the two warps of a sub-partition share the B rows evenly) and eight
  // channel chunks; the two half-warps' chunks sit 16 channels apart (no bank conflicts on G).
  uint8_t* sAS = sm + kOffAS;
  {
    const int chh = warp >> 2, J = chh == 0 ? (warp & 3) : 3 - (warp & 3);
    const int lh = lane >> 4, j = 16 * J + (lane & 15), r = 16 * J;
    const bool vj = j < len;
    const float rk = s_rk[j], rq = s_rq[j];
#pragma unroll 1
    for (int it = 0; it < 4; ++it) {
      const int c16 = 8 * chh + (it & 1) + 4 * (it >> 1) + 2 * lh, c0 = 8 * c16;
      float kf[8], qf[8], kd[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(sK + sw128_offset(j, c0, kC, 2)), kf);
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(sQ + sw128_offset(j, c0, kC, 2)), qf);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float d = sG[j * kGP + c0 + e] - sG[r * kGP + c0 + e];
        const float P = __expf(d), kr = rk * kf[e];
        kd[e] = vj ? kr * __expf(-d) : 0.f;
        kf[e] = vj ? to_tf32(kr * P) : 0.f;
        qf[e] = vj ? to_tf32(rq * qf[e] * P) : 0.f;
      }
      put_tf32x8(sAS, 2 * kC, j, c0, kf);
      put_tf32x8(sAS, 2 * kC, kC + j, c0, qf);
#pragma unroll
      for (int e = 0; e < 8; ++e) kf[e] = to_tf32(kd[e]);
      put_tf32x8(sm + b_off(J), 16 * (J + 1), j, c0, kf);
      for (int I = J + 1; I < 4; ++I) {
        const float4* t4 = reinterpret_cast<const float4*>(&s_T[I * (I - 1) / 2 + J][c0]);
        const float4 ta = t4[0], tb4 = t4[1];
        const float t[8] = {ta.x, ta.y, ta.z, ta.w, tb4.x, tb4.y, tb4.z, tb4.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) kf[e] = to_tf32(t[e] * kd[e]);
        put_tf32x8(sm + b_off(I), 16 * (I + 1), j, c0, kf);
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const uint32_t as = smem_u32(sAS);
    for (int I = 0; I < 4; ++I) {
      const uint32_t n = 16 * (I + 1), bs = smem_u32(sm + b_off(I));
      const uint32_t id_g = idesc_tf32(128, int(n));
      for (int s = 0; s < 16; ++s)
        mma_tf32_ss(tb + I * 64, desc_kmajor(as, 16384, s), desc_kmajor(bs, n * 128u, s), id_g, s > 0);
    }
    mma_commit(&bar_mma);
  }
  __syncwarp();
  // While the Gram products run: the per-token outputs that need only q, k and G. Thread
  // (c, hf) takes channel c of the 32 tokens from 32 hf; Qt, Kt and G leave as coalesced rows,
  // Qt^T and Kt^T as this thread's own row segments.
  {
    const int c = tid & 127, t0 = 32 * hf;
    const float glc = s_gl[c];
    if (hf == 0) p.gam[tile * kD + c] = expf(glc);
    const size_t tw = tile * kTileW;
#pragma unroll 1
    for (int g8 = 0; g8 < 4; ++g8) {
      float qv[8], kv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int t = t0 + 8 * g8 + e;
        const bool vt = t < len;
        const float G = sG[t * kGP + c];
        qv[e] = vt ? to_tf32(p.scale * s_rq[t] * __expf(G) * bf16_at(sQ, t, c)) : 0.f;
        kv[e] = vt ? to_tf32(s_rk[t] * __expf(glc - G) * bf16_at(sK, t, c)) : 0.f;
        const size_t o = tw + size_t(t) * kD + c;
        p.Qt[o] = qv[e];
        if (p.Kt) p.Kt[o] = kv[e];
        if (p.Gc) p.Gc[(tile * kC + t) * kD + c] = G;
      }
      const size_t ot = tile * kTileKtT + size_t(c) * kC + t0 + 8 * g8;
      st_f32x8(p.KtT + ot, kv);
      if (p.QtT) st_f32x8(p.QtT + ot, qv);
    }
    if (tid < kC) {
      if (p.rq) p.rq[tile * kC + tid] = s_rq[tid];
      if (p.rk) p.rk[tile * kC + tid] = s_rk[tid];
      if (p.beff) p.beff[tile * kC + tid] = s_b[tid];
    }
  }
  bool ok = mbar_wait(&bar_mma, 0, &abort_flag, p.status, kDevTimeoutMma);
  uint32_t mma_phase = 1;
  tc_fence_after();
  if (tid == 0 && ok) {
    // the products have read B_1 out of the value tile's slot: load the values there now
    mbar_expect_tx(&bar_v, 16384u);
    for (int pp = 0; pp < 2; ++pp) tma_load_2d(sV + pp * 8192, &mv, h * kD + 64 * pp, ch.x, &bar_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // Row blocks of L (lanes 0..63) and Aqk (lanes 64..127) from D_I, I = block of the row; the
  // two halves of the block take 32 columns j each. Aqk rows are staged (padded [64][65]) and
  // leave as whole lines, row-major and transposed.
  float* sLT = reinterpret_cast<float*>(sm + kOffLT);
  float* sAqk = reinterpret_cast<float*>(sm + kOffAqkS);
  if (ok) {
    const int row = tid & 127, i = row & 63, j0 = 32 * hf;
    const bool isq = row >= kC;
    // The lanes of one warp cover two row blocks (I0, I0 + 1); the TMEM load address must be
    // warp-uniform, so load both and select per lane.
    const int I0 = 2 * (warp & 1);
    const bool second = ((i >> 4) & 1) != 0;
    float r0[32], r1[32];
    tmem_ld32(tl + I0 * 64 + j0, r0);
    tmem_ld32(tl + (I0 + 1) * 64 + j0, r1);
    tmem_wait_ld_regs(r0);
    tmem_wait_ld_regs(r1);
    const bool vi = i < len;
    if (!isq) {
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int j = j0 + jj;
        sLT[j * kC + i] = (j < i && vi) ? s_b[i] * (second ? r1[jj] : r0[jj]) : 0.f;
      }
    } else {
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const int j = j0 + jj;
        sAqk[i * kAP + j] = (j <= i && vi) ? to_tf32(p.scale * (second ? r1[jj] : r0[jj])) : 0.f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  float* sX = reinterpret_cast<float*>(sm + kOffX);
  if (hf == 0) {
    // warps 0-3: A = (I + L)^-1, one column per lane pair
    unit_lower_inverse_column(sLT, sX, 16 * warp + (lane & 15), lane >> 4);
  } else {
    // warps 4-7 meanwhile: K1T = (k (.) exp(G))^T (tf32, K-major [c][j]) in the B region, which
    // the Gram products have released. Thread (token j, chunk group) takes eight channels at a
    // time from one 16-byte key load; the lanes' consecutive tokens make each transposed store
    // one line.
    const int j = lane + 32 * (warp & 1), cg = (warp >> 1) & 1;
    const bool vj = j < len;
#pragma unroll 1
    for (int it = 0; it < 8; ++it) {
      const int c0 = 8 * (8 * cg + it);
      float kf[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(sK + sw128_offset(j, c0, kC, 2)), kf);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        put32(sm + kOffK1T, kD, c0 + e, j, vj ? to_tf32(kf[e] * __expf(sG[j * kGP + c0 + e])) : 0.f);
    }
  }
  __syncthreads();
  // WY operands: A1 = (A - I) diag(beta r_k) (tf32), A2 = (A - I) diag(beta) (bf16), both
  // K-major [i][j]; four threads per column j, 16 rows each. The value tile has landed by now;
  // its rows past the chunk are cleared first.
  ok = ok && mbar_wait(&bar_v, 0, &abort_flag, p.status, kDevTimeoutTma);
  if (ok && tid >= len && tid < kC) {
    for (int c16 = 0; c16 < 16; ++c16)
      *reinterpret_cast<uint4*>(sV + sw128_offset(tid, c16 * 8, kC, 2)) = make_uint4(0, 0, 0, 0);
  }
  {
    const int j = tid & 63, i0 = 16 * (tid >> 6);
    const float s1 = s_b[j] * s_rk[j], s2 = s_b[j];
#pragma unroll 4
    for (int i = i0; i < i0 + 16; ++i) {
      const float x = i == j ? 0.f : sX[i * kC + j];
      put32(sm + kOffA1, kC, i, j, to_tf32(x * s1));
      *reinterpret_cast<__nv_bfloat16*>(sm + kOffA2 + sw128_offset(i, j, kC, 2)) = __float2bfloat16_rn(x * s2);
    }
    if (p.A) {
      float* a = p.A + tile * kTileAqk + j;
      for (int i = i0; i < i0 + 16; ++i) a[size_t(i) * kC] = sX[i * kC + j];
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The WY products transposed, so that the accumulator lanes are channels: W^T = K1^T A1^T
  // (tf32) and U^T = V^T A2^T (bf16, the value tile read MN-major), 128 lanes by 64 tokens.
  if (tid == 0 && ok) {
    const uint32_t a1 = smem_u32(sm + kOffA1), a2 = smem_u32(sm + kOffA2), k1t = smem_u32(sm + kOffK1T);
    const uint32_t v0 = smem_u32(sV);
    const uint32_t idw = idesc_tf32(128, 64), idu = idesc_bf16(128, 64, true, false);
    for (int s = 0; s < 8; ++s) mma_tf32_ss(tb, desc_kmajor(k1t, 16384, s), desc_kmajor(a1, 8192, s), idw, s > 0);
    for (int s = 0; s < 4; ++s) mma_bf16_ss(tb + 128, desc_mnmajor_bf16(v0, 8192, s), desc_kmajor(a2, 8192, s), idu, s > 0);
    mma_commit(&bar_mma);
  }
  // Aqk and its transpose leave from their staging (beside K1T, untouched since the Gram
  // epilogue) while the products run.
  if (ok) {
    float* aqk = p.Aqk + tile * kTileAqk;
#pragma unroll 4
    for (int m = 0; m < kC * kC / kThreads; ++m) {
      const int idx = m * kThreads + tid, r = idx >> 6, col = idx & 63;
      aqk[idx] = sAqk[r * kAP + col];
      if (p.AqkT) p.AqkT[tile * kTileAqk + idx] = sAqk[col * kAP + r];  // (r, col) of Aqk^T
    }
  }
  __syncwarp();
  ok = ok && mbar_wait(&bar_mma, mma_phase, &abort_flag, p.status, kDevTimeoutMma);
  tc_fence_after();
  // W and U rows: thread (c, hf) takes channel c of the 32 tokens from 32 hf, with the unit
  // diagonal of A added in fp32: W = A1 K1 + beta r_k exp(G) k and U = A2 v + beta v. W and U
  // leave as coalesced rows, W^T as this thread's own row segments.
  {
    const int c = tid & 127, t0 = 32 * hf;
    float xw[32], xu[32];
    if (ok) {
      tmem_ld32(tl + t0, xw);
      tmem_ld32(tl + 128 + t0, xu);
      tmem_wait_ld_regs(xw);
      tmem_wait_ld_regs(xu);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) xw[i] = xu[i] = 0.f;
    }
    const size_t tw = tile * kTileW;
#pragma unroll
    for (int g8 = 0; g8 < 4; ++g8) {
      float wv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int t = t0 + 8 * g8 + e;
        const bool vt = t < len;
        const float E = __expf(sG[t * kGP + c]);
        wv[e] = vt ? to_tf32(fmaf(s_b[t] * s_rk[t] * E, bf16_at(sK, t, c), xw[8 * g8 + e])) : 0.f;
        const float u = vt ? fmaf(s_b[t], bf16_at(sV, t, c), xu[8 * g8 + e]) : 0.f;
        const size_t o = tw + size_t(t) * kD + c;
        p.W[o] = wv[e];
        p.U[o] = u;
      }
      if (p.WT) st_f32x8(p.WT + tile * kTileKtT + size_t(c) * kC + t0 + 8 * g8, wv);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 256);
}

cudaError_t launch_prep_kda(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const PrepParams& p, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_prep_kda, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(unsigned(p.NC) * unsigned(p.hgn));
  k_prep_kda<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace gdn
