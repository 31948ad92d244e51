// Gradients of the in-kernel KDA gate parameters (the safe gate of the KDA page's
// `_prepare_kda`: lower_bound * sigmoid(exp(A_log[h]) (x + dt_bias[h][k]))), returned like
// `chunk_kda_bwd_finalize`'s `da_log` and `ddt_bias`.
//
// The token-major backward leaves one partial sum per (chunk, head, channel): ddt_part is the
// sum over the chunk's tokens of dx, dA_part the sum of dg lb s (1 - s) z. Here one CTA per
// head sums them over the chunks (thread k walks the chunks of channel k in order, so
// consecutive threads read consecutive addresses) and reduces dA over the channels in a fixed
// tree, so the result does not depend on scheduling.
#include "common.cuh"

namespace gdn {

__global__ void __launch_bounds__(kD) k_gate_grad(const GateGradParams p) {
  __shared__ float s_a[kD];
  const int h = blockIdx.x, k = threadIdx.x;
  float a = 0.f, d = 0.f;
  for (int c = 0; c < p.NC; ++c) {
    const size_t o = (size_t(c) * p.H + h) * kD + k;
    a += p.dA_part[o];
    d += p.ddt_part[o];
  }
  p.ddt_bias[h * kD + k] = d;
  s_a[k] = a;
  __syncthreads();
  for (int w = kD / 2; w > 0; w >>= 1) {
    if (k < w) s_a[k] += s_a[k + w];
    __syncthreads();
  }
  if (k == 0) p.dA_log[h] = s_a[0];
}

cudaError_t launch_gate_grad(const GateGradParams& p, cudaStream_t s) {
  k_gate_grad<<<p.H, kD, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
