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
// GB300 mapping: the columns of E are independent, so each (sequence, head) is split over
// kColBlocks CTAs of kCols columns, and the walk runs on the CUDA cores in fp32 (a 128x128x16
// product per step and CTA, about a microsecond; the tensor-core version needed three
// split-tf32 products to keep fp32 accuracy and ran on N*H CTAs only). M_s arrives transposed
// (row j = column j of M, as the map runs write it) by one bulk copy per step into a double
// buffer, so the next step's map is in flight while this step computes; the CTA's columns of
// E stay in shared memory between steps. Thread t computes rows 4 (t / 8) .. +3 and columns
// 2 (t % 8), +1 of the block. All waits bounded; every exit decision is taken CTA-wide.
#include "common.cuh"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kCols = 16;                      // columns of E per CTA
constexpr int kColBlocks = kD / kCols;         // CTAs per (sequence, head)
constexpr uint32_t kMapBytes = kD * kD * 4;    // one transposed map, [j][k] fp32
constexpr uint32_t kOffM = 0;                  // two map buffers
constexpr uint32_t kOffE = 2 * kMapBytes;      // [128][kCols] fp32: the current E block
constexpr uint32_t kSmemBytes = kOffE + kD * kCols * 4 + 16;

}  // namespace

__global__ void __launch_bounds__(kThreads, 1) k_compose(const ComposeParams p) {
  extern __shared__ __align__(16) uint8_t smem_c[];
  __shared__ uint64_t full[2];
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int n = blockIdx.x / kColBlocks, cb = blockIdx.x % kColBlocks;
  const int h = blockIdx.y + p.hg0, H = p.H;
  const SegPlan& sp = p.sp;
  const int ns = (p.seqs[n].y + sp.L - 1) / sp.L;
  if (ns < 3) return;  // nothing between the fully-run first segment and pass 1
  const size_t slot_base = size_t(n) * sp.maxS;
  auto slot = [&](int s) { return (slot_base + s) * H + h; };
  float* sE = reinterpret_cast<float*>(smem_c + kOffE);
  const int c0 = cb * kCols;                         // first column of this CTA
  const int k0 = 4 * (tid >> 3), vp = 2 * (tid & 7);  // this thread's rows and column pair

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_mbar_init();
    mbar_expect_tx(&full[0], kMapBytes);
    bulk_load(smem_c + kOffM, sp.Phi + slot(1) * kD * kD, kMapBytes, &full[0]);
  }
  // E[1] columns c0 .. c0 + kCols - 1 (row j: 16 floats, two threads of a row per 32 bytes)
  for (int i = tid; i < kD * kCols / 4; i += kThreads) {
    const int j = i / (kCols / 4), q4 = i % (kCols / 4);
    reinterpret_cast<float4*>(sE)[i] =
        *reinterpret_cast<const float4*>(sp.E + slot(1) * kD * kD + size_t(j) * kD + c0 + 4 * q4);
  }
  __syncthreads();
#pragma unroll 1
  for (int s = 1; s <= ns - 2; ++s) {
    const int buf = (s - 1) & 1;
    // the offset rows of this step, requested before the map is waited for
    const float* Bs = sp.Bm + slot(s) * kD * kD + size_t(k0) * kD + c0 + vp;
    float acc[4][2];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float2 b = *reinterpret_cast<const float2*>(Bs + size_t(kk) * kD);
      acc[kk][0] = b.x;
      acc[kk][1] = b.y;
    }
    const bool ok = mbar_wait(&full[buf], ((s - 1) >> 1) & 1, &abort_flag, p.status, kDevTimeoutTma);
    if (__syncthreads_or(!ok)) {
      // the only copy that can be in flight is this step's (the next one is issued after a
      // successful wait): let it land before the CTA's shared memory goes
      if (tid == 0) mbar_drain(&full[buf], ((s - 1) >> 1) & 1);
      break;
    }
    // the next step's map into the other buffer (its last readers finished the previous step)
    if (tid == 0 && s + 1 <= ns - 2) {
      mbar_expect_tx(&full[buf ^ 1], kMapBytes);
      bulk_load(smem_c + kOffM + (buf ^ 1) * kMapBytes, sp.Phi + slot(s + 1) * kD * kD, kMapBytes, &full[buf ^ 1]);
    }
    // E[s+1] = M_s E[s] + B_s for rows k0..k0+3, columns vp, vp+1 of the block
    const float* Mt = reinterpret_cast<const float*>(smem_c + kOffM + buf * kMapBytes);
#pragma unroll 4
    for (int j = 0; j < kD; ++j) {
      const float4 m = *reinterpret_cast<const float4*>(Mt + j * kD + k0);   // M[k0..k0+3][j]
      const float2 e = *reinterpret_cast<const float2*>(sE + j * kCols + vp);
      acc[0][0] = fmaf(m.x, e.x, acc[0][0]);
      acc[0][1] = fmaf(m.x, e.y, acc[0][1]);
      acc[1][0] = fmaf(m.y, e.x, acc[1][0]);
      acc[1][1] = fmaf(m.y, e.y, acc[1][1]);
      acc[2][0] = fmaf(m.z, e.x, acc[2][0]);
      acc[2][1] = fmaf(m.z, e.y, acc[2][1]);
      acc[3][0] = fmaf(m.w, e.x, acc[3][0]);
      acc[3][1] = fmaf(m.w, e.y, acc[3][1]);
    }
    __syncthreads();  // every thread has read E[s]
    float* dst = sp.E + slot(s + 1) * kD * kD + size_t(k0) * kD + c0 + vp;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float2 r = make_float2(acc[kk][0], acc[kk][1]);
      *reinterpret_cast<float2*>(sE + (k0 + kk) * kCols + vp) = r;
      *reinterpret_cast<float2*>(dst + size_t(kk) * kD) = r;
    }
    __syncthreads();
  }
}

cudaError_t launch_compose(const ComposeParams& p, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_compose, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(p.N * kColBlocks, p.hgn);
  k_compose<<<grid, kThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
