// Host side of libgdn: contract validation, workspace layout, TMA descriptors and the launch
// sequence of every entry point declared in include/gdn.h.
//
// Contract (the interface of the pages' native GDN/KDA adapters, restated): BSND inputs,
// K == V == 128, chunk size 64; packed documents only with batch size 1 and a host offsets
// array that starts at 0, strictly increases and ends at T (zero-length documents are
// rejected); a contract violation is a GDN_EINVAL error raised before any work is enqueued
// (the adapters' ValueError), an unsupported device a GDN_EUNSUPPORTED error (their
// RuntimeError).
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "gdn.h"

namespace gdn {
namespace {

thread_local std::string g_err;

int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D row-major tensor: `cols` contiguous elements per row, `rows` rows `stride_bytes` apart.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t cols, uint64_t rows,
              uint64_t stride_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {stride_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Problem {
  int B, T, H, N, NC, R;
  float scale;
  bool packed;
  std::vector<int32_t> cu;  // packed offsets (host copy)
};

int validate_desc(const gdn_desc_t* d, Problem* P) {
  if (!d) return fail(GDN_EINVAL, "desc is NULL");
  if (d->K != kD || d->V != kD) return fail(GDN_EINVAL, "K and V must both be 128");
  if (d->chunk_size != kC) return fail(GDN_EINVAL, "chunk_size must be 64");
  if (d->B < 1 || d->T < 1 || d->H < 1) return fail(GDN_EINVAL, "B, T and H must be positive");
  if (std::isnan(d->scale) || std::isinf(d->scale)) return fail(GDN_EINVAL, "scale must be finite");
  P->B = d->B;
  P->T = d->T;
  P->H = d->H;
  P->scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt(float(d->K));
  P->packed = d->cu_seqlens != nullptr;
  const long long R = (long long)d->B * d->T;
  if (R > (1ll << 30)) return fail(GDN_EINVAL, "B*T too large");
  P->R = int(R);
  long long NC = 0;
  if (P->packed) {
    if (d->B != 1) return fail(GDN_EINVAL, "packed documents (cu_seqlens) require batch size 1");
    if (d->num_seqs < 1) return fail(GDN_EINVAL, "num_seqs must be >= 1 with cu_seqlens");
    const int32_t* cu = d->cu_seqlens;
    if (cu[0] != 0) return fail(GDN_EINVAL, "cu_seqlens must start at 0");
    for (int i = 0; i < d->num_seqs; ++i) {
      if (cu[i + 1] <= cu[i]) return fail(GDN_EINVAL, "cu_seqlens must be strictly increasing (no empty documents)");
      NC += (cu[i + 1] - cu[i] + kC - 1) / kC;
    }
    if (cu[d->num_seqs] != d->T) return fail(GDN_EINVAL, "cu_seqlens must end at T");
    P->N = d->num_seqs;
    P->cu.assign(cu, cu + d->num_seqs + 1);
  } else {
    P->N = d->B;
    NC = (long long)d->B * ((d->T + kC - 1) / kC);
  }
  if (NC * d->H * kD >= (1ll << 31)) return fail(GDN_EINVAL, "problem too large for 32-bit tile coordinates");
  P->NC = int(NC);
  return GDN_OK;
}

struct FwdLayout {
  size_t cu, seqs, chunks, W, U, Qt, KtT, Aqk, gam, total;
};

FwdLayout fwd_layout(const Problem& P) {
  FwdLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const size_t tiles = size_t(P.NC) * P.H;
  L.cu = take(sizeof(int) * (P.N + 1));
  L.seqs = take(sizeof(SeqEntry) * P.N);
  L.chunks = take(sizeof(ChunkEntry) * P.NC);
  L.W = take(4 * tiles * kTileW);
  L.U = take(4 * tiles * kTileW);
  L.Qt = take(4 * tiles * kTileW);
  L.KtT = take(4 * tiles * kTileKtT);
  L.Aqk = take(4 * tiles * kTileAqk);
  L.gam = take(4 * tiles * kD);
  L.total = off;
  return L;
}

int device_check() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(GDN_EUNSUPPORTED, "no CUDA device");
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return fail(GDN_EUNSUPPORTED, "device is not compute capability 10.3 (GB300)");
  return GDN_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b) return false;
  const char* pa = static_cast<const char*>(a);
  const char* pb = static_cast<const char*>(b);
  return pa < pb + nb && pb < pa + na;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_cuda(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(GDN_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return GDN_OK;
}

// Copy the packed offsets into the workspace through kernel parameters (no host staging
// buffer outlives the call), then build the chunk and sequence tables on the device.
int build_tables(const Problem& P, void* ws, const FwdLayout& L, int* status, cudaStream_t s) {
  char* base = static_cast<char*>(ws);
  int* dcu = nullptr;
  if (P.packed) {
    dcu = reinterpret_cast<int*>(base + L.cu);
    const int total = P.N + 1;
    for (int off = 0; off < total; off += kMaxUploadInts) {
      UploadParams up;
      up.count = std::min(kMaxUploadInts, total - off);
      for (int i = 0; i < up.count; ++i) up.vals[i] = P.cu[off + i];
      int rc = check_cuda(launch_upload(up, dcu + off, s), "upload offsets");
      if (rc) return rc;
    }
  }
  TableParams tp;
  tp.cu = dcu;
  tp.N = P.N;
  tp.T = P.T;
  tp.NC = P.NC;
  tp.seqs = reinterpret_cast<SeqEntry*>(base + L.seqs);
  tp.chunks = reinterpret_cast<ChunkEntry*>(base + L.chunks);
  tp.status = status;
  return check_cuda(launch_tables(tp, s), "chunk tables");
}

int run_fwd(const gdn_desc_t* d, const gdn_fwd_args_t* a, void* stream, bool kda) {
  Problem P;
  int rc = validate_desc(d, &P);
  if (rc) return rc;
  if (!a) return fail(GDN_EINVAL, "args is NULL");
  if (!a->q || !a->k || !a->v || !a->g || !a->beta || !a->o)
    return fail(GDN_EINVAL, "q, k, v, g, beta and o must be non-NULL");
  if (d->output_final_state && !a->final_state) return fail(GDN_EINVAL, "final_state is NULL but requested");
  if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v))
    return fail(GDN_EINVAL, "q, k and v must be 16-byte aligned");
  const size_t nqk = size_t(P.R) * P.H * kD * 2;
  if (overlaps(a->o, nqk, a->q, nqk) || overlaps(a->o, nqk, a->k, nqk) || overlaps(a->o, nqk, a->v, nqk))
    return fail(GDN_EINVAL, "o must not alias q, k or v");
  const FwdLayout L = fwd_layout(P);
  if (!a->workspace || a->workspace_bytes < L.total)
    return fail(GDN_EINVAL, "workspace missing or smaller than the required size");
  if (reinterpret_cast<uintptr_t>(a->workspace) & 255) return fail(GDN_EINVAL, "workspace must be 256-byte aligned");
  if (kda) return fail(GDN_EUNSUPPORTED, "per-channel gate forward is not built yet");
  rc = device_check();
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(a->workspace);

  rc = build_tables(P, ws, L, a->status, s);
  if (rc) return rc;

  CUtensorMap mq, mk, mv, mW, mQt, mKtT, mAqk, mU;
  const uint64_t HD = uint64_t(P.H) * kD;
  const uint64_t rows64 = uint64_t(P.NC) * P.H * kC, rows128 = uint64_t(P.NC) * P.H * kD;
  bool ok = make_map(&mq, a->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, HD, P.R, HD * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&mk, a->k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, HD, P.R, HD * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&mv, a->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, HD, P.R, HD * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&mW, ws + L.W, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, kD, rows64, kD * 4, 32, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&mQt, ws + L.Qt, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, kD, rows64, kD * 4, 32, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&mU, ws + L.U, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, kD, rows64, kD * 4, 32, 64, CU_TENSOR_MAP_SWIZZLE_NONE) &&
            make_map(&mKtT, ws + L.KtT, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, kC, rows128, kC * 4, 32, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&mAqk, ws + L.Aqk, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, kC, rows64, kC * 4, 32, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return fail(GDN_ECUDA, "cuTensorMapEncodeTiled failed");

  PrepParams pp{};
  pp.chunks = reinterpret_cast<const ChunkEntry*>(ws + L.chunks);
  pp.NC = P.NC;
  pp.H = P.H;
  pp.g = a->g;
  pp.beta = static_cast<const __nv_bfloat16*>(a->beta);
  pp.scale = P.scale;
  pp.l2norm = d->use_qk_l2norm;
  pp.beta_sigmoid = d->use_beta_sigmoid;
  pp.W = reinterpret_cast<float*>(ws + L.W);
  pp.U = reinterpret_cast<float*>(ws + L.U);
  pp.Qt = reinterpret_cast<float*>(ws + L.Qt);
  pp.KtT = reinterpret_cast<float*>(ws + L.KtT);
  pp.Aqk = reinterpret_cast<float*>(ws + L.Aqk);
  pp.gam = reinterpret_cast<float*>(ws + L.gam);
  pp.status = a->status;
  rc = check_cuda(launch_prep_gdn(mq, mk, mv, pp, s), "prepare kernel");
  if (rc) return rc;

  ChainParams cp{};
  cp.seqs = reinterpret_cast<const SeqEntry*>(ws + L.seqs);
  cp.chunks = pp.chunks;
  cp.N = P.N;
  cp.H = P.H;
  cp.kda = 0;
  cp.gam = pp.gam;
  cp.h0 = a->initial_state;
  cp.hT = d->output_final_state ? a->final_state : nullptr;
  cp.o = static_cast<__nv_bfloat16*>(a->o);
  cp.status = a->status;
  return check_cuda(launch_chain_fwd(mW, mQt, mKtT, mAqk, mU, cp, s), "chain kernel");
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

const char* gdn_strerror(int code) {
  switch (code) {
    case GDN_OK: return "success";
    case GDN_EINVAL: return "invalid argument (contract violation)";
    case GDN_EUNSUPPORTED: return "unsupported device or feature";
    case GDN_ECUDA: return "CUDA runtime error";
    case GDN_ETIMEOUT: return "bounded device wait expired";
    default: return "unknown error";
  }
}

const char* gdn_last_error(void) { return g_err.c_str(); }

int gdn_device_supported(int device) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess)
    return fail(GDN_EUNSUPPORTED, "no such CUDA device");
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
  return (major == 10 && minor == 3) ? GDN_OK : GDN_EUNSUPPORTED;
}

size_t gdn_fwd_workspace_size(const gdn_desc_t* desc) {
  Problem P;
  if (validate_desc(desc, &P)) return 0;
  return fwd_layout(P).total;
}

size_t kda_fwd_workspace_size(const gdn_desc_t* desc) { return gdn_fwd_workspace_size(desc); }

size_t gdn_bwd_workspace_size(const gdn_desc_t* desc) {
  Problem P;
  if (validate_desc(desc, &P)) return 0;
  return 0;
}

size_t kda_bwd_workspace_size(const gdn_desc_t* desc) { return gdn_bwd_workspace_size(desc); }

int gdn_fwd(const gdn_desc_t* desc, const gdn_fwd_args_t* args, void* stream) {
  g_err.clear();
  return run_fwd(desc, args, stream, false);
}

int kda_fwd(const gdn_desc_t* desc, const gdn_fwd_args_t* args, void* stream) {
  g_err.clear();
  return run_fwd(desc, args, stream, true);
}

int gdn_bwd(const gdn_desc_t* desc, const gdn_bwd_args_t* args, void* stream) {
  (void)desc; (void)args; (void)stream;
  return fail(GDN_EUNSUPPORTED, "backward is not built yet");
}

int kda_bwd(const gdn_desc_t* desc, const gdn_bwd_args_t* args, void* stream) {
  (void)desc; (void)args; (void)stream;
  return fail(GDN_EUNSUPPORTED, "backward is not built yet");
}

}  // extern "C"
