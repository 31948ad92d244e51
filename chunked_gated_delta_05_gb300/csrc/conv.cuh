// Parameters of the causal depthwise convolution kernels (k_conv.cu).
#pragma once
#include "common.cuh"

namespace gdn {

constexpr int kConvMaxTaps = 8;

struct ConvParams {
  const __nv_bfloat16* x;      // [R,C]
  const float* w;              // [C,W]: tap i multiplies x[t - (W-1-i) dil]
  const float* bias;           // [C] or null
  const __nv_bfloat16* halo;   // [N,HW,C] inputs before each sequence's first row, or null (zeros)
  __nv_bfloat16* y;            // [R,C]
  const __nv_bfloat16* dy;     // backward: [R,C]
  __nv_bfloat16* dx;           // backward: [R,C]
  float* dz;                   // backward workspace: [R,C] fp32
  float* part;                 // backward workspace: [tiles,C,W+1] partial sums
  float *dw, *dbias;           // backward outputs [C,W], [C] (dbias may be null)
  float* dhalo;                // backward output [N,HW,C] fp32, or null
  const int* cu;               // device copy of the sequence offsets, or null (dense)
  long long R;                 // rows (B*T)
  int T, N, C, W, dil, HW;     // HW = (W-1) dil halo rows
  int silu;
};

cudaError_t launch_conv_fwd(const ConvParams& p, cudaStream_t s);
cudaError_t launch_conv_bwd(const ConvParams& p, cudaStream_t s);
size_t conv_partials_bytes(long long R, int C, int W);

}  // namespace gdn
