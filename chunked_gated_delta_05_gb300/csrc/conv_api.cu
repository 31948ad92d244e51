// Host side of the short convolution: contract validation, workspace layout and launches of
// gdn_conv_fwd / gdn_conv_bwd (declared in include/gdn.h).
#include <cstdio>
#include <vector>

#include "conv.cuh"
#include "gdn.h"

namespace gdn {
namespace {

struct ConvProblem {
  long long R;
  int B, T, C, W, dil, N, HW;
  bool packed;
  std::vector<int32_t> cu;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int validate_conv(const gdn_conv_desc_t* d, ConvProblem* P) {
  if (!d) return set_last_error(GDN_EINVAL, "desc is NULL");
  if (d->B < 1 || d->T < 1 || d->C < 8 || d->C % 8) return set_last_error(GDN_EINVAL, "B, T >= 1 and C a positive multiple of 8 required");
  if (d->W < 1 || d->W > kConvMaxTaps) return set_last_error(GDN_EINVAL, "W must be 1..8");
  if (d->dilation < 1) return set_last_error(GDN_EINVAL, "dilation must be >= 1");
  if (d->activation != 0 && d->activation != 1) return set_last_error(GDN_EINVAL, "activation must be 0 or 1");
  P->B = d->B;
  P->T = d->T;
  P->C = d->C;
  P->W = d->W;
  P->dil = d->dilation;
  P->HW = (d->W - 1) * d->dilation;
  P->R = (long long)d->B * d->T;
  if (P->R * d->C >= (1ll << 40)) return set_last_error(GDN_EINVAL, "problem too large");
  P->packed = d->cu_seqlens != nullptr;
  if (P->packed) {
    if (d->B != 1) return set_last_error(GDN_EINVAL, "packed documents (cu_seqlens) require batch size 1");
    if (d->num_seqs < 1) return set_last_error(GDN_EINVAL, "num_seqs must be >= 1 with cu_seqlens");
    const int32_t* cu = d->cu_seqlens;
    if (cu[0] != 0) return set_last_error(GDN_EINVAL, "cu_seqlens must start at 0");
    for (int i = 0; i < d->num_seqs; ++i)
      if (cu[i + 1] <= cu[i]) return set_last_error(GDN_EINVAL, "cu_seqlens must be strictly increasing");
    if (cu[d->num_seqs] != d->T) return set_last_error(GDN_EINVAL, "cu_seqlens must end at T");
    P->N = d->num_seqs;
    P->cu.assign(cu, cu + d->num_seqs + 1);
  } else {
    P->N = d->B;
  }
  return GDN_OK;
}

struct ConvLayout {
  size_t cu, dz, part, total;
};

ConvLayout conv_layout(const ConvProblem& P, bool backward) {
  ConvLayout L{};
  size_t off = 0;
  L.cu = off;
  off = align256(off + sizeof(int) * (P.N + 1));
  if (backward) {
    L.dz = off;
    off = align256(off + size_t(P.R) * P.C * 4);
    L.part = off;
    off = align256(off + conv_partials_bytes(P.R, P.C, P.W));
  }
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int device_ok() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return set_last_error(GDN_EUNSUPPORTED, "no CUDA device");
  if (gdn_device_supported(dev) != GDN_OK)
    return set_last_error(GDN_EUNSUPPORTED, "device is not compute capability 10.3 (GB300)");
  return GDN_OK;
}

int cuda_rc(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return GDN_OK;
  char msg[256];
  snprintf(msg, sizeof(msg), "%s: %s", what, cudaGetErrorString(e));
  return set_last_error(GDN_ECUDA, msg);
}

int prepare(const ConvProblem& P, char* ws, const ConvLayout& L, ConvParams* cp, cudaStream_t s) {
  cp->R = P.R;
  cp->T = P.T;
  cp->N = P.N;
  cp->C = P.C;
  cp->W = P.W;
  cp->dil = P.dil;
  cp->HW = P.HW;
  cp->cu = nullptr;
  if (P.packed) {
    int* dcu = reinterpret_cast<int*>(ws + L.cu);
    int rc = upload_offsets(P.cu.data(), P.N + 1, dcu, s);
    if (rc) return rc;
    cp->cu = dcu;
  }
  return GDN_OK;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

size_t gdn_conv_fwd_workspace_size(const gdn_conv_desc_t* desc) {
  ConvProblem P;
  if (validate_conv(desc, &P)) return 0;
  return conv_layout(P, false).total;
}

size_t gdn_conv_bwd_workspace_size(const gdn_conv_desc_t* desc) {
  ConvProblem P;
  if (validate_conv(desc, &P)) return 0;
  return conv_layout(P, true).total;
}

int gdn_conv_fwd(const gdn_conv_desc_t* desc, const gdn_conv_fwd_args_t* a, void* stream) {
  ConvProblem P;
  int rc = validate_conv(desc, &P);
  if (rc) return rc;
  if (!a || !a->x || !a->weight || !a->y) return set_last_error(GDN_EINVAL, "x, weight and y must be non-NULL");
  if (!aligned16(a->x) || !aligned16(a->y) || (a->halo && !aligned16(a->halo)) || !aligned16(a->weight) ||
      (a->bias && !aligned16(a->bias)))
    return set_last_error(GDN_EINVAL, "x, y, halo, weight and bias must be 16-byte aligned");
  const size_t bytes = size_t(P.R) * P.C * 2;
  const char *xb = static_cast<const char*>(a->x), *yb = static_cast<const char*>(a->y);
  if (xb < yb + bytes && yb < xb + bytes) return set_last_error(GDN_EINVAL, "y must not alias x");
  const ConvLayout L = conv_layout(P, false);
  if (!a->workspace || a->workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(a->workspace) & 255))
    return set_last_error(GDN_EINVAL, "workspace missing, too small or not 256-byte aligned");
  if ((rc = device_ok())) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ConvParams cp{};
  if ((rc = prepare(P, static_cast<char*>(a->workspace), L, &cp, s))) return rc;
  cp.x = static_cast<const __nv_bfloat16*>(a->x);
  cp.w = a->weight;
  cp.bias = a->bias;
  cp.halo = static_cast<const __nv_bfloat16*>(a->halo);
  cp.y = static_cast<__nv_bfloat16*>(a->y);
  cp.silu = desc->activation;
  TimedScope t(kKConvFwd, s);
  return cuda_rc(launch_conv_fwd(cp, s), "convolution kernel");
}

int gdn_conv_bwd(const gdn_conv_desc_t* desc, const gdn_conv_bwd_args_t* a, void* stream) {
  ConvProblem P;
  int rc = validate_conv(desc, &P);
  if (rc) return rc;
  if (!a || !a->x || !a->weight || !a->dy || !a->dx || !a->dweight)
    return set_last_error(GDN_EINVAL, "x, weight, dy, dx and dweight must be non-NULL");
  if (!aligned16(a->x) || !aligned16(a->dy) || !aligned16(a->dx) || (a->halo && !aligned16(a->halo)) ||
      (a->dhalo && !aligned16(a->dhalo)) || !aligned16(a->weight) || (a->bias && !aligned16(a->bias)))
    return set_last_error(GDN_EINVAL, "x, dy, dx, halo, dhalo, weight and bias must be 16-byte aligned");
  if (a->dhalo && !a->halo) return set_last_error(GDN_EINVAL, "dhalo needs the halo input");
  const size_t bytes = size_t(P.R) * P.C * 2;
  const char* dxb = static_cast<const char*>(a->dx);
  for (const void* in : {a->x, a->dy}) {
    const char* ib = static_cast<const char*>(in);
    if (dxb < ib + bytes && ib < dxb + bytes) return set_last_error(GDN_EINVAL, "dx must not alias x or dy");
  }
  const ConvLayout L = conv_layout(P, true);
  if (!a->workspace || a->workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(a->workspace) & 255))
    return set_last_error(GDN_EINVAL, "workspace missing, too small or not 256-byte aligned");
  if ((rc = device_ok())) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(a->workspace);
  ConvParams cp{};
  if ((rc = prepare(P, ws, L, &cp, s))) return rc;
  cp.x = static_cast<const __nv_bfloat16*>(a->x);
  cp.w = a->weight;
  cp.bias = a->bias;
  cp.halo = static_cast<const __nv_bfloat16*>(a->halo);
  cp.dy = static_cast<const __nv_bfloat16*>(a->dy);
  cp.dx = static_cast<__nv_bfloat16*>(a->dx);
  cp.dz = reinterpret_cast<float*>(ws + L.dz);
  cp.part = reinterpret_cast<float*>(ws + L.part);
  cp.dw = a->dweight;
  cp.dbias = a->dbias;
  cp.dhalo = a->dhalo;
  cp.silu = desc->activation;
  TimedScope t(kKConvBwd, s);
  return cuda_rc(launch_conv_bwd(cp, s), "convolution backward kernels");
}

}  // extern "C"
