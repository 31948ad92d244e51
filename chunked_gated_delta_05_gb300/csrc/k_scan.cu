// Compose kernel of the segmented chain: walks one sequence's segments in processing order,
//   E[s+1] = M_s E[s] + B_s,        s = 1 .. ns-2,
// where (M_s, B_s) is segment s's affine state map from the chain's map runs and E[1] the
// exit state of the fully-run segment 0. The maps are the per-chunk summaries
// state_out = M state_in + S, M = e^{g_last} I - (k e^{g_last - g})^T w, S = (k e^{g_last - g})^T u,
// composed over a segment's chunks, that the pages' context-parallel GDN path builds per rank
// and applies to the incoming state (hyper-parallel GDN Diff Coverage page,
// `_compute_gdn_state_summary_from_prepared` and `_apply_gdn_state_summary`; the backward's
// adjoint summary, grad_in = M^T grad_out + G, is `apply_kda_state_gradient_summary` on the
// Ascend GDN Diff Coverage page). Here the "ranks" are segments of one sequence on one GPU,
// and the reverse chain's adjoint maps compose the same way.
//
// GB300 mapping: one CTA of 128 threads per (sequence, head). E^T lives in TMEM (lane v =
// column v of E) as two tf32 parts, E_hi + E_lo; M arrives by TMA as its two tf32 parts
// (K-major SW128 B operands) together with B_s (the next step's copies are issued as soon as
// the MMAs are done, under the epilogue); the product is accumulated in TMEM on top of B_s^T with three
// tf32 MMA groups, E_hi M_hi + E_lo M_hi + E_hi M_lo, so the composition keeps fp32 accuracy
// (split-tf32 products; the dropped E_lo M_lo term is below fp32 rounding). Thread 0 issues
// the copies and the MMAs. All waits bounded; every exit decision is taken CTA-wide.
#include "common.cuh"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 128;
constexpr uint32_t kMapBytes = 65536;        // one 128 x 128 fp32 map part: 4 panels x 128 rows x 128 B
constexpr uint32_t kOffHi = 0, kOffLo = kMapBytes, kOffB = 2 * kMapBytes;  // B: 4 plain [128][32] panels
constexpr uint32_t kSmemBytes = 3 * kMapBytes + 1024;
constexpr uint32_t kTD = 0, kTEH = 128, kTEL = 256;

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    k_compose(const __grid_constant__ CUtensorMap mPhi, const __grid_constant__ CUtensorMap mPlo,
              const __grid_constant__ CUtensorMap mB, const ComposeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1k(smem_raw);
  __shared__ uint64_t full, mma;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int n = blockIdx.x, h = blockIdx.y + p.hg0, H = p.H;
  const SegPlan& sp = p.sp;
  const int ns = (p.seqs[n].y + sp.L - 1) / sp.L;
  if (ns < 3) return;  // nothing between the fully-run first segment and pass 1
  const size_t slot_base = size_t(n) * sp.maxS;
  auto slot = [&](int s) { return (slot_base + s) * H + h; };
  // copies of step s: both parts of M_s (swizzled K-major B operands) and B_s (plain panels)
  auto issue = [&](int s) {
    const int y = int(slot(s)) * kD;
    mbar_expect_tx(&full, 3 * kMapBytes);
    for (int pp = 0; pp < 4; ++pp) {
      tma_load_2d(sm + kOffHi + pp * 16384, &mPhi, pp * 32, y, &full);
      tma_load_2d(sm + kOffLo + pp * 16384, &mPlo, pp * 32, y, &full);
      tma_load_2d(sm + kOffB + pp * 16384, &mB, pp * 32, y, &full);
    }
  };

  if (warp == 0) tmem_alloc(&tslot, 512);
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&full, 1);
    mbar_init(&mma, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  const uint32_t tl = tb + tmem_lane_base(warp);
  const int v = tid;
  const uint32_t sHi = smem_u32(sm + kOffHi), sLo = smem_u32(sm + kOffLo);
  const float* sBm = reinterpret_cast<const float*>(sm + kOffB) + (v >> 5) * 4096 + (v & 31);

  if (tid == 0) {
    issue(1);
    // the later maps start their trip to L2 now (the walk is serial)
    for (int s = 2; s <= ns - 2; ++s) {
      prefetch_l2(sp.Phi + slot(s) * kD * kD, 4u * kD * kD);
      prefetch_l2(sp.Plo + slot(s) * kD * kD, 4u * kD * kD);
      prefetch_l2(sp.Bm + slot(s) * kD * kD, 4u * kD * kD);
    }
  }
  // E[1]^T row v, split into its tf32 parts
  {
    const float* src = sp.E + slot(1) * kD * kD + v;
#pragma unroll 1
    for (int g = 0; g < 4; g += 2) {
      float x[64];
#pragma unroll
      for (int e = 0; e < 64; ++e) x[e] = src[size_t(32 * g + e) * kD];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float hi[32], lo[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          hi[e] = to_tf32(x[32 * hh + e]);
          lo[e] = to_tf32(x[32 * hh + e] - hi[e]);
        }
        tmem_st32(tl + kTEH + 32 * (g + hh), hi);
        tmem_st32(tl + kTEL + 32 * (g + hh), lo);
      }
    }
  }
  const uint32_t id = idesc_tf32(128, 128);
#pragma unroll 1
  for (int s = 1; s <= ns - 2; ++s) {
    const uint32_t par = (s - 1) & 1;
    bool ok = mbar_wait(&full, par, &abort_flag, p.status, kDevTimeoutTma);
    if (ok) {
      // accumulator <- B_s^T (lane v = column v of B_s), from the staged plain panels
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        float b[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) b[e] = sBm[(32 * g + e) * 32];
        tmem_st32(tl + kTD + 32 * g, b);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    if (__syncthreads_or(!ok)) break;
    if (tid == 0) {
      tc_fence_after();
      for (int k = 0; k < 16; ++k) mma_tf32_ts(tb + kTD, tb + kTEH + k * 8, desc_kmajor(sHi, 16384, k), id, true);
      for (int k = 0; k < 16; ++k) mma_tf32_ts(tb + kTD, tb + kTEL + k * 8, desc_kmajor(sHi, 16384, k), id, true);
      for (int k = 0; k < 16; ++k) mma_tf32_ts(tb + kTD, tb + kTEH + k * 8, desc_kmajor(sLo, 16384, k), id, true);
      mma_commit(&mma);
    }
    ok = mbar_wait(&mma, par, &abort_flag, p.status, kDevTimeoutMma);
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();
    // the next step's copies overlap this step's epilogue (the MMAs no longer read the tiles)
    if (tid == 0 && s + 1 <= ns - 2) issue(s + 1);
    // E[s+1]^T row v: store it, and split it into the next step's operand
    {
      float* dst = sp.E + slot(s + 1) * kD * kD + v;
#pragma unroll 1
      for (int g = 0; g < 4; ++g) {
        float r[32];
        tmem_ld32(tl + kTD + 32 * g, r);
        tmem_wait_ld_regs(r);
        float lo[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          dst[size_t(32 * g + e) * kD] = r[e];
          const float hi = to_tf32(r[e]);
          lo[e] = to_tf32(r[e] - hi);
          r[e] = hi;
        }
        tmem_st32(tl + kTEH + 32 * g, r);
        tmem_st32(tl + kTEL + 32 * g, lo);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 512);
}

cudaError_t launch_compose(const CUtensorMap& mPhi, const CUtensorMap& mPlo, const CUtensorMap& mB,
                           const ComposeParams& p, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_compose, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(p.N, p.hgn);
  k_compose<<<grid, kThreads, kSmemBytes, s>>>(mPhi, mPlo, mB, p);
  return cudaGetLastError();
}

}  // namespace gdn
