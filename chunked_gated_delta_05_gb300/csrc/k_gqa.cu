// Grouped-query heads: H value heads share H / G query/key heads (value head h reads q/k head
// h / G, the pages' `repeat_interleave` of q and k over num_v_heads // num_k_heads, done by
// indexing in the kernels instead of copying). The gradient of a shared q/k head is the sum of
// the gradients its G value heads produce; the token-major backward writes those per value
// head in fp32 and this kernel sums each group in a fixed order (deterministic) and rounds once.
#include "common.cuh"

namespace gdn {

__global__ void __launch_bounds__(256) k_group_sum(const GroupSumParams p) {
  const int Hk = p.H / p.G;
  const long long n4 = p.R * Hk * (kD / 4);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const int d = 4 * int(i % (kD / 4));
    const long long rk = i / (kD / 4);
    const int hk = int(rk % Hk);
    const long long r = rk / Hk;
    float4 aq = make_float4(0.f, 0.f, 0.f, 0.f), ak = aq;
    for (int g = 0; g < p.G; ++g) {
      const size_t src = (size_t(r) * p.H + size_t(hk) * p.G + g) * kD + d;
      const float4 q = __ldg(reinterpret_cast<const float4*>(p.dq32 + src));
      const float4 k = __ldg(reinterpret_cast<const float4*>(p.dk32 + src));
      aq.x += q.x; aq.y += q.y; aq.z += q.z; aq.w += q.w;
      ak.x += k.x; ak.y += k.y; ak.z += k.z; ak.w += k.w;
    }
    const size_t dst = (size_t(r) * Hk + hk) * kD + d;
    __nv_bfloat162* oq = reinterpret_cast<__nv_bfloat162*>(p.dq + dst);
    __nv_bfloat162* ok = reinterpret_cast<__nv_bfloat162*>(p.dk + dst);
    oq[0] = __floats2bfloat162_rn(aq.x, aq.y);
    oq[1] = __floats2bfloat162_rn(aq.z, aq.w);
    ok[0] = __floats2bfloat162_rn(ak.x, ak.y);
    ok[1] = __floats2bfloat162_rn(ak.z, ak.w);
  }
}

cudaError_t launch_group_sum(const GroupSumParams& p, cudaStream_t s) {
  const long long n4 = p.R * (p.H / p.G) * (kD / 4);
  const long long want = (n4 + 255) / 256;
  // a grid-stride loop over at most 16 resident CTAs of 256 threads per SM
  const long long cap = 16ll * (p.sms > 0 ? p.sms : 1);
  const int blocks = int(want < cap ? want : cap);
  k_group_sum<<<blocks > 0 ? blocks : 1, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
