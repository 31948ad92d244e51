// Chain kernel: the serial inter-chunk state recurrence fused with the chunk output.
//
// Per chunk, with S the K x V state entering it (the chunk loop of the eager reference
// `torch_chunk_gated_delta_rule`, hyper-parallel GDN Diff Coverage page):
//   v_new = U - W S
//   o     = Qt S + Aqk v_new
//   S     = gam (.) S + KtT^T-applied: S <- diag(gam) S + (k decayed to chunk end)^T v_new
// (gam is exp(G_last): a scalar for GDN, one value per key row for KDA.)
//
// GB300 mapping: one CTA per (sequence, head). The state is held transposed, S^T (V x K),
// one row per thread of warps 0-3 (thread v owns column v of S, 128 fp32 registers), so
// every product is a 128-lane tcgen05 MMA with S^T or v_new^T as the TMEM-resident A
// operand (kind::tf32; operands rounded to nearest tf32 when written) and the chunk tiles
// from the prepare kernel as TMA-loaded SW128 B operands:
//   P   = S^T  W^T    (v_new^T = U^T - P)        -> TMEM
//   O   = S^T  Qt^T + v_new^T Aqk^T              -> TMEM (double-buffered by chunk parity)
//   D   = v_new^T KtT^T  (= (k~^T v_new)^T)      -> TMEM; S^T <- gam S^T + D in registers
// Warp 4 streams the tiles with TMA (three buffer groups, each refilled as soon as its
// consumers finish) and issues the MMAs from one thread. All waits are bounded.
#include "common.cuh"
#include "umma.cuh"

namespace gdn {

namespace {

constexpr int kThreads = 160;
// shared memory tile offsets (bytes, 1024-aligned)
constexpr uint32_t kOffW = 0;          // 4 panels x 64 rows x 128 B   (W   [t][k], K-major)
constexpr uint32_t kOffQt = 32768;     // 4 panels x 64 rows x 128 B   (Qt  [t][k])
constexpr uint32_t kOffKtT = 65536;    // 2 panels x 128 rows x 128 B  (KtT [k][t])
constexpr uint32_t kOffAqk = 98304;    // 2 panels x 64 rows x 128 B   (Aqk [i][j])
constexpr uint32_t kOffU = 114688;     // 4 panels x [64][32] fp32, no swizzle
constexpr uint32_t kSmemBytes = 147456 + 1024;
// TMEM columns
constexpr uint32_t kTS = 0, kTP = 128, kTVN = 192, kTD = 256, kTO = 384;

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    k_chain_fwd(const __grid_constant__ CUtensorMap mW, const __grid_constant__ CUtensorMap mQt,
                const __grid_constant__ CUtensorMap mKtT, const __grid_constant__ CUtensorMap mAqk,
                const __grid_constant__ CUtensorMap mU, const ChainParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1k(smem_raw);
  __shared__ uint64_t full1, full2, full3, mma1, mma2, sready, vready;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = blockIdx.x, h = blockIdx.y, H = p.H;
  const SeqEntry seq = p.seqs[n];
  const int first = seq.x, nc = seq.y;

  if (warp == 0) tmem_alloc(&tslot, 512);
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&full1, 1);
    mbar_init(&full2, 1);
    mbar_init(&full3, 1);
    mbar_init(&mma1, 1);
    mbar_init(&mma2, 1);
    mbar_init(&sready, 128);
    mbar_init(&vready, 128);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;

  if (warp == 4) {
    if (lane == 0) {
      // ---------------- producer + MMA issuer ----------------
      const uint32_t sW = smem_u32(sm + kOffW), sQt = smem_u32(sm + kOffQt), sKtT = smem_u32(sm + kOffKtT),
                     sAqk = smem_u32(sm + kOffAqk);
      auto load_g1 = [&](int c) {
        const int y = (c * H + h) * kC;
        mbar_expect_tx(&full1, 65536u);
        for (int pp = 0; pp < 4; ++pp) {
          tma_load_2d(sm + kOffW + pp * 8192, &mW, pp * 32, y, &full1);
          tma_load_2d(sm + kOffQt + pp * 8192, &mQt, pp * 32, y, &full1);
        }
      };
      auto load_g2 = [&](int c) {
        const int y = (c * H + h) * kC;
        mbar_expect_tx(&full2, 32768u);
        for (int pp = 0; pp < 4; ++pp) tma_load_2d(sm + kOffU + pp * 8192, &mU, pp * 32, y, &full2);
      };
      auto load_g3 = [&](int c) {
        mbar_expect_tx(&full3, 49152u);
        for (int pp = 0; pp < 2; ++pp) {
          tma_load_2d(sm + kOffKtT + pp * 16384, &mKtT, pp * 32, (c * H + h) * kD, &full3);
          tma_load_2d(sm + kOffAqk + pp * 8192, &mAqk, pp * 32, (c * H + h) * kC, &full3);
        }
      };
      load_g1(first);
      load_g2(first);
      load_g3(first);
      const uint32_t id64 = idesc_tf32(128, 64), id128 = idesc_tf32(128, 128);
      for (int j = 0; j < nc; ++j) {
        const uint32_t par = j & 1;
        const int c = first + j;
        const uint32_t tO = tb + kTO + (j & 1) * 64;
        if (!mbar_wait(&full1, par, &abort_flag, p.status, kDevTimeoutTma)) break;
        if (!mbar_wait(&sready, par, &abort_flag, p.status, kDevTimeoutSync)) break;
        tc_fence_after();
        for (int s = 0; s < 16; ++s) mma_tf32_ts(tb + kTP, tb + kTS + s * 8, desc_kmajor(sW, 8192, s), id64, s > 0);
        for (int s = 0; s < 16; ++s) mma_tf32_ts(tO, tb + kTS + s * 8, desc_kmajor(sQt, 8192, s), id64, s > 0);
        mma_commit(&mma1);
        if (!mbar_wait(&mma1, par, &abort_flag, p.status, kDevTimeoutMma)) break;
        if (j + 1 < nc) load_g1(c + 1);
        if (!mbar_wait(&vready, par, &abort_flag, p.status, kDevTimeoutSync)) break;
        if (j + 1 < nc) load_g2(c + 1);
        if (!mbar_wait(&full3, par, &abort_flag, p.status, kDevTimeoutTma)) break;
        tc_fence_after();
        for (int s = 0; s < 8; ++s) mma_tf32_ts(tO, tb + kTVN + s * 8, desc_kmajor(sAqk, 8192, s), id64, true);
        for (int s = 0; s < 8; ++s) mma_tf32_ts(tb + kTD, tb + kTVN + s * 8, desc_kmajor(sKtT, 16384, s), id128, s > 0);
        mma_commit(&mma2);
        if (!mbar_wait(&mma2, par, &abort_flag, p.status, kDevTimeoutMma)) break;
        if (j + 1 < nc) load_g3(c + 1);
      }
      // Drain: make sure no TMA write is still landing in shared memory before exit.
      // Loads are only issued for chunks that the loop then waits on, except on abort.
    }
  } else {
    // ---------------- chain warps: thread v owns row v of S^T ----------------
    const int v = tid;
    const uint32_t lb = tmem_lane_base(warp);
    const float* sU = reinterpret_cast<const float*>(sm + kOffU);
    float S[kD];
    if (p.h0) {
      const float* src = p.h0 + (size_t(n) * H + h) * kD * kD + v;
#pragma unroll
      for (int k = 0; k < kD; ++k) S[k] = src[size_t(k) * kD];
    } else {
#pragma unroll
      for (int k = 0; k < kD; ++k) S[k] = 0.f;
    }
    auto store_state = [&]() {
#pragma unroll
      for (int c0 = 0; c0 < kD; c0 += 16) {
        float r[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) r[e] = to_tf32(S[c0 + e]);
        tmem_st16(tb + lb + kTS + c0, r);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&sready);
    };
    store_state();
    bool alive = true;
    for (int j = 0; j < nc && alive; ++j) {
      const uint32_t par = j & 1;
      const int c = first + j;
      const ChunkEntry ch = p.chunks[c];
      const size_t tile = size_t(c) * H + h;
      if (p.h_save) {
        float* dst = p.h_save + tile * kD * kD + v;
#pragma unroll
        for (int k = 0; k < kD; ++k) dst[size_t(k) * kD] = S[k];
      }
      if (!mbar_wait(&mma1, par, &abort_flag, p.status, kDevTimeoutMma)) { alive = false; break; }
      tc_fence_after();
      if (!mbar_wait(&full2, par, &abort_flag, p.status, kDevTimeoutTma)) { alive = false; break; }
      // v_new^T row v = U[:, v] - P[v, :]
      float* vsave = p.vnew_save ? p.vnew_save + tile * kTileW + v : nullptr;
#pragma unroll
      for (int t0 = 0; t0 < kC; t0 += 16) {
        float r[16];
        tmem_ld16(tb + lb + kTP + t0, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int t = t0 + e;
          const float u = sU[(v >> 5) * 2048 + t * 32 + (v & 31)];
          const float vn = u - r[e];
          if (vsave) vsave[size_t(t) * kD] = vn;
          r[e] = to_tf32(vn);
        }
        tmem_st16(tb + lb + kTVN + t0, r);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&vready);
      const float* gam = p.gam + tile * kD;  // end-of-chunk decay: entry 0 (GDN) or per key row (KDA)
      const float gsc = gam[0];
      if (!mbar_wait(&mma2, par, &abort_flag, p.status, kDevTimeoutMma)) { alive = false; break; }
      tc_fence_after();
#pragma unroll
      for (int k0 = 0; k0 < kD; k0 += 16) {
        float r[16];
        tmem_ld16(tb + lb + kTD + k0, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float gk = p.kda ? gam[k0 + e] : gsc;
          S[k0 + e] = fmaf(gk, S[k0 + e], r[e]);
        }
      }
      // output rows of this chunk (read before the state is released for the next chunk's
      // MMAs, which may reuse this parity's O buffer two chunks later)
      {
        const uint32_t tO = tb + kTO + (j & 1) * 64;
        __nv_bfloat16* op = p.o ? p.o + (size_t(ch.x) * H + h) * kD + v : nullptr;
#pragma unroll
        for (int t0 = 0; t0 < kC; t0 += 16) {
          float r[16];
          tmem_ld16(tO + lb + t0, r);
          tmem_wait_ld();
          if (op) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int t = t0 + e;
              if (t < ch.y) op[size_t(t) * H * kD] = __float2bfloat16_rn(r[e]);
            }
          }
        }
      }
      store_state();
    }
    if (alive && p.hT) {
      float* dst = p.hT + (size_t(n) * H + h) * kD * kD + v;
#pragma unroll
      for (int k = 0; k < kD; ++k) dst[size_t(k) * kD] = S[k];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 512);
}

cudaError_t launch_chain_fwd(const CUtensorMap& mW, const CUtensorMap& mQt, const CUtensorMap& mKtT,
                             const CUtensorMap& mAqk, const CUtensorMap& mU, const ChainParams& p,
                             cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_chain_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(p.N, p.H);
  k_chain_fwd<<<grid, kThreads, kSmemBytes, s>>>(mW, mQt, mKtT, mAqk, mU, p);
  return cudaGetLastError();
}

}  // namespace gdn
