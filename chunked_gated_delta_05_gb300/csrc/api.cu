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

#include <algorithm>
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
  int Hk, G;                // q/k heads and value heads per q/k head
  float scale;
  bool packed;
  bool gate;                // KDA in-kernel gate activation
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
  if (d->num_k_heads < 0 || (d->num_k_heads > 0 && d->H % d->num_k_heads != 0))
    return fail(GDN_EINVAL, "num_k_heads must be 0 or divide H");
  P->Hk = d->num_k_heads > 0 ? d->num_k_heads : d->H;
  P->G = d->H / P->Hk;
  P->scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt(float(d->K));
  P->gate = d->use_gate_in_kernel != 0;
  if (P->gate && !(d->lower_bound >= -5.f && d->lower_bound < 0.f))
    return fail(GDN_EINVAL, "lower_bound must lie in [-5, 0) with use_gate_in_kernel");
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

// ------------------------------------------------------------------ segmented chain plan
// Segment length (in chunks) forced by gdn_set_chain_segment(); 0 = chosen by plan_scan().
int g_chain_segment = 0;

// Wave model of the chain scan (one chain CTA per SM, waves of sm_count() CTAs): pass 0 runs
// 1 + 2 (ns - 2) CTAs per (sequence, head), pass 1 runs ns - 1, each for about L chunk steps;
// the compose kernel walks ns - 2 segments. The step costs are GB300 measurements (a chain
// step averaged over the forward and reverse chains and over full and map runs under a full
// wave of CTAs; one compose step).
int sm_count();
constexpr double kChunkStepUs = 4.25, kComposeStepUs = 6.0, kLaunchUs = 3.0;
constexpr int kMaxSegments = 64;

struct ScanPlan {
  int L = 1;     // chunks per segment
  int maxS = 1;  // most segments of any sequence
};

ScanPlan plan_scan(const Problem& P) {
  // distinct per-sequence chunk counts with their multiplicities
  std::vector<std::pair<int, int>> lens;
  int maxNC = 0;
  if (P.packed) {
    std::vector<int> nc(P.N);
    for (int n = 0; n < P.N; ++n) nc[n] = (P.cu[n + 1] - P.cu[n] + kC - 1) / kC;
    std::sort(nc.begin(), nc.end());
    for (int x : nc) {
      if (lens.empty() || lens.back().first != x) lens.push_back({x, 0});
      ++lens.back().second;
    }
    maxNC = nc.back();
  } else {
    maxNC = (P.T + kC - 1) / kC;
    lens.push_back({maxNC, P.N});
  }
  auto segments = [&](int L) {
    int m = 0;
    for (auto& e : lens) m = std::max(m, (e.first + L - 1) / L);
    return m;
  };
  ScanPlan best;
  if (g_chain_segment > 0) {
    best.L = std::min(g_chain_segment, maxNC);
    best.maxS = segments(best.L);
    return best;
  }
  double best_t = 1e300;
  const int sms = sm_count();
  for (int S = 1; S <= std::min(maxNC, kMaxSegments); ++S) {
    const int L = (maxNC + S - 1) / S;
    long long runs0 = 0, runs1 = 0;
    int maxS = 0;
    for (auto& e : lens) {
      const int ns = (e.first + L - 1) / L;
      maxS = std::max(maxS, ns);
      runs0 += (long long)e.second * (ns <= 2 ? 1 : 2 * ns - 3);
      runs1 += (long long)e.second * (ns - 1);
    }
    auto waves = [&](long long r) { return double((r * P.H + sms - 1) / sms); };
    double t = waves(runs0) * L * kChunkStepUs;
    if (maxS >= 2) t += waves(runs1) * L * kChunkStepUs + kLaunchUs;
    if (maxS >= 3) t += (maxS - 2) * kComposeStepUs + kLaunchUs;
    if (t < best_t - 1e-9) {
      best_t = t;
      best.L = L;
      best.maxS = maxS;
    }
  }
  return best;
}

// Buffer carve-up. The "saved" part holds the chunk tables, the prepare tiles and (for a
// training forward / backward) the chain saves; the "rest" part holds what only the backward
// uses. Inference forward: saved part only (forward subset). Backward without a saved buffer:
// both parts in the workspace. With a saved buffer: saved part there, rest part in the
// workspace. Every region is 256-byte aligned; rest offsets are relative to the rest base.
struct Layout {
  size_t cu, seqs, chunks, W, U, Qt, KtT, Aqk, gam;               // forward
  size_t Kt, QtT, AqkT, WT, A, Gc, rq, rk, beff;                  // prepare, backward mode
  size_t hs, vns;                                                  // forward chain saves
  size_t fE, fPhi, fB;                                       // forward chain scan (scratch)
  size_t dhs, dvns, dQt, dKt, dW, dK1, dV1, dgam;                  // rest part (relative)
  size_t rE, rPhi, rB;                                       // reverse chain scan (rest part)
  size_t dq32, dk32;                                               // grouped q/k: per-value-head dq, dk
  size_t dA_part, ddt_part;                                        // in-kernel gate: parameter partials
  size_t saved_total, rest_total, total;
  ScanPlan plan;
};

Layout make_layout(const Problem& P, bool backward, bool kda = false) {
  Layout L{};
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
  if (backward) {
    L.Kt = take(4 * tiles * kTileW);
    L.QtT = take(4 * tiles * kTileKtT);
    L.AqkT = take(4 * tiles * kTileAqk);
    L.WT = take(4 * tiles * kTileKtT);
    L.A = take(4 * tiles * kTileAqk);
    L.Gc = take(4 * tiles * kC * (kda ? kD : 1));
    L.rq = take(4 * tiles * kC);
    L.rk = take(4 * tiles * kC);
    L.beff = take(4 * tiles * kC);
    L.hs = take(2 * tiles * kD * kD);   // bf16
    L.vns = take(4 * tiles * kTileW);
  }
  L.plan = plan_scan(P);
  const size_t scan_states = L.plan.maxS > 1 ? size_t(P.N) * L.plan.maxS * P.H * kD * kD * 4 : 0;
  L.fE = take(scan_states);
  L.fPhi = take(scan_states);
  L.fB = take(scan_states);
  L.saved_total = off;
  off = 0;
  if (backward) {
    L.dhs = take(2 * tiles * kD * kD);  // bf16
    L.dvns = take(4 * tiles * kTileW);
    L.dQt = take(2 * tiles * kTileW);   // bf16
    L.dKt = take(2 * tiles * kTileW);   // bf16
    L.dW = take(4 * tiles * kTileW);
    L.dK1 = take(2 * tiles * kTileW);   // bf16
    L.dV1 = take(4 * tiles * kTileW);
    L.dgam = take(4 * tiles * kD);
    L.rE = take(scan_states);
    L.rPhi = take(scan_states);
    L.rB = take(scan_states);
    const size_t per_head = P.G > 1 ? size_t(P.R) * P.H * kD * 4 : 0;
    L.dq32 = take(per_head);
    L.dk32 = take(per_head);
    const size_t gate_parts = P.gate ? 4 * tiles * kD : 0;
    L.dA_part = take(gate_parts);
    L.ddt_part = take(gate_parts);
  }
  L.rest_total = off;
  L.total = L.saved_total + L.rest_total;
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

// SM count of the current device (a prefetch distance for the chunk kernels).
int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 152;  // a GB300's SM count
  return n > 0 ? n : 152;
}

int check_cuda(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(GDN_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return GDN_OK;
}

// Optional per-kernel timing (CUDA events recorded on the launching stream around every
// launch while enabled). Process-global and not thread-safe: a profiling aid.
const char* const kKindNames[kKinds] = {"tables", "prepare", "chain_fwd", "chain_bwd", "bwd_feat", "bwd_tok",
                                        "compose", "group_sum", "conv_fwd", "conv_bwd", "gate_grad"};
struct Timing {
  bool on = false;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev[kKinds];
  size_t used[kKinds] = {};
} g_tim;

struct TimedLaunch {
  int kind;
  cudaStream_t s;
  bool active;
  TimedLaunch(int k, cudaStream_t st) : kind(k), s(st), active(g_tim.on) {
    if (!active) return;
    auto& v = g_tim.ev[kind];
    if (g_tim.used[kind] == v.size()) {
      cudaEvent_t a, b;
      cudaEventCreate(&a);
      cudaEventCreate(&b);
      v.push_back({a, b});
    }
    cudaEventRecord(v[g_tim.used[kind]].first, s);
  }
  ~TimedLaunch() {
    if (!active) return;
    cudaEventRecord(g_tim.ev[kind][g_tim.used[kind]].second, s);
    ++g_tim.used[kind];
  }
};

struct Maps {
  CUtensorMap q, k, v, W, Qt, KtT, Aqk, U, Usw;      // forward (Usw: U as a swizzled store target)
  CUtensorMap Kt, AqkT, QtT, WT, VN, DVN, DW, dO;     // backward
  CUtensorMap Hs, DHs;                               // saved states h, dh' [tile][128][128] bf16 (128-row boxes)
};

// Row-major fp32 workspace tiles as TMA sources: `cols` per row, boxes of 32 columns.
bool tile_map(CUtensorMap* m, const char* base, uint64_t cols, uint64_t rows, uint32_t box_rows, bool swz) {
  return make_map(m, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, cols, rows, cols * 4, 32, box_rows,
                  swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

// The bf16 state saves h, dh' [tile][128][128] as TMA sources: 128-row boxes of 64 columns
// (128 bytes, one 128-byte swizzle panel).
bool state_map(CUtensorMap* m, const char* base, uint64_t rows) {
  return make_map(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kD, rows, kD * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Whether the layout carries the backward-mode prepare tiles.
bool backward_tiles(const Layout& L) { return L.Kt != 0; }

bool fwd_maps(const Problem& P, const void* q, const void* k, const void* v, const char* ws, const Layout& L, Maps* M) {
  const uint64_t HD = uint64_t(P.H) * kD, HDk = uint64_t(P.Hk) * kD;
  const uint64_t r64 = uint64_t(P.NC) * P.H * kC, r128 = uint64_t(P.NC) * P.H * kD;
  return make_map(&M->q, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, HDk, P.R, HDk * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(&M->k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, HDk, P.R, HDk * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(&M->v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, HD, P.R, HD * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
         tile_map(&M->W, ws + L.W, kD, r64, 64, true) && tile_map(&M->Qt, ws + L.Qt, kD, r64, 64, true) &&
         tile_map(&M->U, ws + L.U, kD, r64, 64, false) && tile_map(&M->Usw, ws + L.U, kD, r64, 64, true) &&
         tile_map(&M->KtT, ws + L.KtT, kC, r128, 128, true) && tile_map(&M->Aqk, ws + L.Aqk, kC, r64, 64, true) &&
         (!backward_tiles(L) || tile_map(&M->Kt, ws + L.Kt, kD, r64, 64, true));
}

bool bwd_maps(const Problem& P, const char* sv, const char* rs, const Layout& L, Maps* M) {
  const uint64_t r64 = uint64_t(P.NC) * P.H * kC, r128 = uint64_t(P.NC) * P.H * kD;
  return tile_map(&M->Kt, sv + L.Kt, kD, r64, 64, true) && tile_map(&M->AqkT, sv + L.AqkT, kC, r64, 64, true) &&
         tile_map(&M->QtT, sv + L.QtT, kC, r128, 128, true) && tile_map(&M->WT, sv + L.WT, kC, r128, 128, true) &&
         tile_map(&M->VN, sv + L.vns, kD, r64, 64, true) && tile_map(&M->DVN, rs + L.dvns, kD, r64, 64, true) &&
         tile_map(&M->DW, rs + L.dW, kD, r64, 64, true) && state_map(&M->Hs, sv + L.hs, r128) && state_map(&M->DHs, rs + L.dhs, r128);
}

// Prepare-kernel parameters for a buffer carved by make_layout at `sv` (backward-mode outputs
// only when `backward`).
PrepParams prep_params(const gdn_desc_t* d, const Problem& P, char* sv, const Layout& L, const float* g,
                       const void* beta, bool backward, int* status, const float* A_log, const float* dt_bias) {
  auto F = [&](size_t off) { return reinterpret_cast<float*>(sv + off); };
  PrepParams pp{};
  pp.chunks = reinterpret_cast<const ChunkEntry*>(sv + L.chunks);
  pp.NC = P.NC;
  pp.dense_T = P.packed ? 0 : P.T;
  pp.H = P.H;
  pp.g = g;
  pp.beta = static_cast<const __nv_bfloat16*>(beta);
  pp.scale = P.scale;
  pp.l2norm = d->use_qk_l2norm;
  pp.beta_sigmoid = d->use_beta_sigmoid;
  pp.qk_group = P.G;
  pp.W = F(L.W); pp.U = F(L.U); pp.Qt = F(L.Qt); pp.KtT = F(L.KtT); pp.Aqk = F(L.Aqk); pp.gam = F(L.gam);
  if (backward) {
    pp.Gc = F(L.Gc); pp.rq = F(L.rq); pp.rk = F(L.rk); pp.beff = F(L.beff);
    pp.Kt = F(L.Kt); pp.QtT = F(L.QtT); pp.AqkT = F(L.AqkT); pp.WT = F(L.WT); pp.A = F(L.A);
  }
  pp.gate_act = P.gate ? 1 : 0;
  pp.lower_bound = d->lower_bound;
  pp.A_log = A_log;
  pp.dt_bias = dt_bias;
  pp.status = status;
  return pp;
}

// Copy the packed offsets into the workspace through kernel parameters (no host staging
// buffer outlives the call), then build the chunk and sequence tables on the device.
int build_tables(const Problem& P, void* ws, const Layout& L, int* status, cudaStream_t s) {
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
  TimedLaunch tl_(kKTables, s);
  return check_cuda(launch_tables(tp, s), "chunk tables");
}

SegPlan seg_plan(const ScanPlan& sc, char* base, size_t E, size_t Phi, size_t B) {
  SegPlan sp{};
  sp.L = sc.L;
  sp.maxS = sc.maxS;
  sp.pass = 0;
  sp.E = reinterpret_cast<float*>(base + E);
  sp.Phi = reinterpret_cast<float*>(base + Phi);
  sp.Bm = reinterpret_cast<float*>(base + B);
  return sp;
}

// ------------------------------------------------------------------ head groups
// A large problem splits its heads into two groups: the first runs on the caller's stream, the
// second on a stream the library keeps per device, forked after the work already enqueued on
// the caller's stream and joined back into it before the call returns, so the call keeps its
// single-stream ordering. The two groups' kernels share the SMs, and the low-occupancy phases
// of one group (the chain's second pass, the compose step) overlap the other group's work.
// Every kernel computes each head independently, so the results do not depend on the grouping.
int g_head_groups = 0;  // forced number of groups (1 or 2), 0 = automatic
constexpr int kMaxDevices = 64;
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;
SideStream g_side[kMaxDevices];

// Automatic choice, from GB300 measurements of both forms on the benchmark workloads: the
// backward gains from 1024 chunk-heads on, the forward from 4096 (below that its prepare and
// chain passes already fill the GPU and the split only adds launches).
int wanted_groups(const Problem& P, bool backward) {
  if (g_head_groups > 0) return std::min(std::min(g_head_groups, 2), P.H);
  const size_t chunk_heads = size_t(P.NC) * P.H;
  return (P.H >= 8 && chunk_heads >= (backward ? 1024u : 4096u)) ? 2 : 1;
}

class HeadGroups {
 public:
  HeadGroups(const Problem& P, bool backward, cudaStream_t s) : s_(s), H_(P.H), n_(wanted_groups(P, backward)) {
    if (n_ < 2) return;
    lock_ = std::unique_lock<std::mutex>(g_side_mu);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
      n_ = 1;
      return;
    }
    SideStream& ss = g_side[dev];
    if (!ss.s) {
      if (cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess ||
          cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess) {
        n_ = 1;
        return;
      }
    }
    if (cudaEventRecord(ss.fork, s) != cudaSuccess || cudaStreamWaitEvent(ss.s, ss.fork, 0) != cudaSuccess) {
      n_ = 1;
      return;
    }
    side_ = &ss;
  }
  ~HeadGroups() { join(); }
  int count() const { return n_; }
  int first(int g) const { return n_ == 1 ? 0 : (g == 0 ? 0 : H_ / 2); }
  int heads(int g) const { return n_ == 1 ? H_ : (g == 0 ? H_ / 2 : H_ - H_ / 2); }
  cudaStream_t stream(int g) const { return g == 0 ? s_ : side_->s; }
  // The caller's stream waits for the second group (idempotent).
  int join() {
    if (!side_) return GDN_OK;
    SideStream* ss = side_;
    side_ = nullptr;
    if (cudaEventRecord(ss->join, ss->s) != cudaSuccess || cudaStreamWaitEvent(s_, ss->join, 0) != cudaSuccess)
      return fail(GDN_ECUDA, "joining the head-group stream failed");
    return GDN_OK;
  }

 private:
  cudaStream_t s_;
  int H_, n_;
  SideStream* side_ = nullptr;
  std::unique_lock<std::mutex> lock_;
};

// Compose step between the two chain passes (sequences with three or more segments), for the
// heads hg0 .. hg0 + hgn - 1.
int run_compose(const Problem& P, const SeqEntry* seqs, const SegPlan& sp, int* status, int hg0, int hgn,
                cudaStream_t s) {
  ComposeParams cp{};
  cp.seqs = seqs;
  cp.N = P.N;
  cp.H = P.H;
  cp.hg0 = hg0;
  cp.hgn = hgn;
  cp.sp = sp;
  cp.status = status;
  TimedLaunch tl_(kKCompose, s);
  return check_cuda(launch_compose(cp, s), "compose kernel");
}

// Forward chain: one plain pass, or pass 0, compose, pass 1 of the segmented chain.
int run_chain_fwd(const Problem& P, const Maps& M, ChainParams cp, cudaStream_t s) {
  for (int pass = 0; pass < (cp.sp.maxS > 1 ? 2 : 1); ++pass) {
    if (pass == 1 && cp.sp.maxS >= 3) {
      int rc = run_compose(P, cp.seqs, cp.sp, cp.status, cp.hg0, cp.hgn, s);
      if (rc) return rc;
    }
    cp.sp.pass = pass;
    TimedLaunch tl_(kKChainFwd, s);
    int rc = check_cuda(launch_chain_fwd(M.W, M.Qt, M.KtT, M.Aqk, M.U, cp, s), "chain kernel");
    if (rc) return rc;
  }
  return GDN_OK;
}

// Reverse chain, same structure.
int run_chain_bwd(const Problem& P, const Maps& M, RevChainParams rp, cudaStream_t s) {
  for (int pass = 0; pass < (rp.sp.maxS > 1 ? 2 : 1); ++pass) {
    if (pass == 1 && rp.sp.maxS >= 3) {
      int rc = run_compose(P, rp.seqs, rp.sp, rp.status, rp.hg0, rp.hgn, s);
      if (rc) return rc;
    }
    rp.sp.pass = pass;
    TimedLaunch tl_(kKChainBwd, s);
    int rc = check_cuda(launch_chain_bwd(M.Kt, M.AqkT, M.QtT, M.WT, M.dO, rp, s), "reverse chain kernel");
    if (rc) return rc;
  }
  return GDN_OK;
}

int run_fwd(const gdn_desc_t* d, const gdn_fwd_args_t* a, void* stream, bool kda) {
  Problem P;
  int rc = validate_desc(d, &P);
  if (rc) return rc;
  if (!a) return fail(GDN_EINVAL, "args is NULL");
  if (!a->q || !a->k || !a->v || !a->g || !a->beta || !a->o)
    return fail(GDN_EINVAL, "q, k, v, g, beta and o must be non-NULL");
  if (d->output_final_state && !a->final_state) return fail(GDN_EINVAL, "final_state is NULL but requested");
  if (P.gate && !kda) return fail(GDN_EINVAL, "use_gate_in_kernel is a KDA option (the GDN gate comes in activated)");
  if (P.gate && (!a->A_log || !a->dt_bias)) return fail(GDN_EINVAL, "use_gate_in_kernel needs A_log and dt_bias");
  if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->o))
    return fail(GDN_EINVAL, "q, k, v and o must be 16-byte aligned");
  const size_t nqk = size_t(P.R) * P.Hk * kD * 2, nv = size_t(P.R) * P.H * kD * 2;
  if (overlaps(a->o, nv, a->q, nqk) || overlaps(a->o, nv, a->k, nqk) || overlaps(a->o, nv, a->v, nv))
    return fail(GDN_EINVAL, "o must not alias q, k or v");
  const bool training = a->saved != nullptr;
  const Layout L = make_layout(P, training, kda);
  char* ws = nullptr;
  if (training) {
    if (a->saved_bytes < L.saved_total) return fail(GDN_EINVAL, "saved buffer smaller than the required size");
    if (reinterpret_cast<uintptr_t>(a->saved) & 255) return fail(GDN_EINVAL, "saved buffer must be 256-byte aligned");
    ws = static_cast<char*>(a->saved);
  } else {
    if (!a->workspace || a->workspace_bytes < L.saved_total)
      return fail(GDN_EINVAL, "workspace missing or smaller than the required size");
    if (reinterpret_cast<uintptr_t>(a->workspace) & 255) return fail(GDN_EINVAL, "workspace must be 256-byte aligned");
    ws = static_cast<char*>(a->workspace);
  }
  rc = device_check();
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  rc = build_tables(P, ws, L, a->status, s);
  if (rc) return rc;
  Maps M;
  if (!fwd_maps(P, a->q, a->k, a->v, ws, L, &M)) return fail(GDN_ECUDA, "cuTensorMapEncodeTiled failed");
  PrepParams pp = prep_params(d, P, ws, L, a->g, a->beta, training, a->status, a->A_log, a->dt_bias);
  ChainParams cp{};
  cp.seqs = reinterpret_cast<const SeqEntry*>(ws + L.seqs);
  cp.chunks = pp.chunks;
  cp.N = P.N;
  cp.H = P.H;
  cp.kda = kda ? 1 : 0;
  cp.gam = pp.gam;
  cp.h0 = a->initial_state;
  cp.hT = d->output_final_state ? a->final_state : nullptr;
  cp.o = static_cast<__nv_bfloat16*>(a->o);
  if (training) {
    cp.h_save = reinterpret_cast<__nv_bfloat16*>(ws + L.hs);
    cp.vnew_save = reinterpret_cast<float*>(ws + L.vns);
  }
  cp.status = a->status;
  cp.sp = seg_plan(L.plan, ws, L.fE, L.fPhi, L.fB);
  HeadGroups groups(P, false, s);
  for (int g = 0; g < groups.count(); ++g) {
    const cudaStream_t sg = groups.stream(g);
    pp.hg0 = cp.hg0 = groups.first(g);
    pp.hgn = cp.hgn = groups.heads(g);
    {
      TimedLaunch tl_(kKPrep, sg);
      rc = check_cuda(kda ? launch_prep_kda(M.q, M.k, M.v, pp, sg)
                          : launch_prep_gdn(M.q, M.k, M.v, M.Qt, training ? M.Kt : M.Qt, M.Aqk, M.W, M.Usw, pp, sg),
                      "prepare kernel");
    }
    if (rc) return rc;
    rc = run_chain_fwd(P, M, cp, sg);
    if (rc) return rc;
  }
  return groups.join();
}

int run_bwd(const gdn_desc_t* d, const gdn_bwd_args_t* a, void* stream, bool kda) {
  Problem P;
  int rc = validate_desc(d, &P);
  if (rc) return rc;
  if (!a) return fail(GDN_EINVAL, "args is NULL");
  if (!a->q || !a->k || !a->v || !a->g || !a->beta || !a->dO || !a->dq || !a->dk || !a->dv || !a->dbeta || !a->dg)
    return fail(GDN_EINVAL, "q, k, v, g, beta, dO and every gradient output except dh0 must be non-NULL");
  if (P.gate && !kda) return fail(GDN_EINVAL, "use_gate_in_kernel is a KDA option (the GDN gate comes in activated)");
  if (P.gate && (!a->A_log || !a->dt_bias || !a->dA_log || !a->ddt_bias))
    return fail(GDN_EINVAL, "use_gate_in_kernel needs A_log, dt_bias, dA_log and ddt_bias");
  if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->dO) || !aligned16(a->dq) ||
      !aligned16(a->dk) || !aligned16(a->dv))
    return fail(GDN_EINVAL, "q, k, v, dO, dq, dk and dv must be 16-byte aligned");
  const size_t nqk = size_t(P.R) * P.Hk * kD * 2, nv = size_t(P.R) * P.H * kD * 2;
  const void* ins[] = {a->q, a->k, a->v, a->dO};
  const size_t in_bytes[] = {nqk, nqk, nv, nv};
  const void* outs[] = {a->dq, a->dk, a->dv};
  const size_t out_bytes[] = {nqk, nqk, nv};
  for (int oi = 0; oi < 3; ++oi)
    for (int ii = 0; ii < 4; ++ii)
      if (overlaps(outs[oi], out_bytes[oi], ins[ii], in_bytes[ii]))
        return fail(GDN_EINVAL, "gradient outputs must not alias the inputs");
  const Layout L = make_layout(P, true, kda);
  const bool have_saved = a->saved != nullptr;
  if (have_saved) {
    if (a->saved_bytes < L.saved_total) return fail(GDN_EINVAL, "saved buffer smaller than the required size");
    if (reinterpret_cast<uintptr_t>(a->saved) & 255) return fail(GDN_EINVAL, "saved buffer must be 256-byte aligned");
  }
  const size_t need = have_saved ? L.rest_total : L.total;
  if (!a->workspace || a->workspace_bytes < need)
    return fail(GDN_EINVAL, "workspace missing or smaller than the required size");
  if (reinterpret_cast<uintptr_t>(a->workspace) & 255) return fail(GDN_EINVAL, "workspace must be 256-byte aligned");
  rc = device_check();
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* sv = have_saved ? const_cast<char*>(static_cast<const char*>(a->saved)) : static_cast<char*>(a->workspace);
  char* rs = have_saved ? static_cast<char*>(a->workspace) : static_cast<char*>(a->workspace) + L.saved_total;
  Maps M;
  const uint64_t HD = uint64_t(P.H) * kD;
  if (!fwd_maps(P, a->q, a->k, a->v, sv, L, &M) || !bwd_maps(P, sv, rs, L, &M) ||
      !make_map(&M.dO, a->dO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, HD, P.R, HD * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return fail(GDN_ECUDA, "cuTensorMapEncodeTiled failed");
  auto F = [&](size_t off) { return reinterpret_cast<float*>(sv + off); };
  auto R = [&](size_t off) { return reinterpret_cast<float*>(rs + off); };
  auto H16 = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(rs + off); };
  const ChunkEntry* chunks = reinterpret_cast<const ChunkEntry*>(sv + L.chunks);
  PrepParams pp{};
  ChainParams cp{};
  if (have_saved) {
    // the forward already built the tables and saved its intermediates; reset the status word
    if (a->status) {
      rc = check_cuda(cudaMemsetAsync(a->status, 0, sizeof(int), s), "status reset");
      if (rc) return rc;
    }
  } else {
    rc = build_tables(P, sv, L, a->status, s);
    if (rc) return rc;
    pp = prep_params(d, P, sv, L, a->g, a->beta, true, a->status, a->A_log, a->dt_bias);
    cp.seqs = reinterpret_cast<const SeqEntry*>(sv + L.seqs);
    cp.chunks = chunks;
    cp.kda = kda ? 1 : 0;
    cp.N = P.N;
    cp.H = P.H;
    cp.gam = F(L.gam);
    cp.h0 = a->initial_state;
    cp.h_save = reinterpret_cast<__nv_bfloat16*>(sv + L.hs);
    cp.vnew_save = F(L.vns);
    cp.status = a->status;
    cp.sp = seg_plan(L.plan, sv, L.fE, L.fPhi, L.fB);
  }

  RevChainParams rp{};
  rp.seqs = reinterpret_cast<const SeqEntry*>(sv + L.seqs);
  rp.chunks = chunks;
  rp.N = P.N;
  rp.H = P.H;
  rp.gam = F(L.gam);
  rp.kda = kda ? 1 : 0;
  rp.dO = static_cast<const __nv_bfloat16*>(a->dO);
  rp.dht = a->dht;
  rp.dh0 = a->dh0;
  rp.dh_save = reinterpret_cast<__nv_bfloat16*>(rs + L.dhs);
  rp.dvn_save = R(L.dvns);
  rp.status = a->status;
  rp.sp = seg_plan(L.plan, rs, L.rE, L.rPhi, L.rB);

  BwdFeatParams fp{};
  fp.chunks = chunks;
  fp.NC = P.NC;
  fp.dense_T = P.packed ? 0 : P.T;
  fp.H = P.H;
  fp.kda = kda ? 1 : 0;
  fp.h = reinterpret_cast<const __nv_bfloat16*>(sv + L.hs);
  fp.dh = reinterpret_cast<const __nv_bfloat16*>(rs + L.dhs);
  fp.dO = rp.dO;
  fp.A = F(L.A);
  fp.dvn = R(L.dvns);
  fp.dQt = H16(L.dQt); fp.dKt = H16(L.dKt); fp.dW = R(L.dW); fp.dK1 = H16(L.dK1); fp.dV1 = R(L.dV1);
  fp.dgam = R(L.dgam);
  fp.sms = sm_count();
  fp.status = a->status;

  BwdTokParams tp{};
  tp.chunks = chunks;
  tp.NC = P.NC;
  tp.dense_T = P.packed ? 0 : P.T;
  tp.H = P.H;
  tp.scale = P.scale;
  tp.beta_sigmoid = d->use_beta_sigmoid;
  tp.l2norm = d->use_qk_l2norm;
  tp.dO = rp.dO;
  tp.A = F(L.A);
  tp.Gc = F(L.Gc); tp.rq = F(L.rq); tp.rk = F(L.rk); tp.beff = F(L.beff);
  tp.dQt = H16(L.dQt); tp.dKt = H16(L.dKt); tp.dK1 = H16(L.dK1); tp.dV1 = R(L.dV1);
  tp.gam = F(L.gam); tp.dgam = R(L.dgam);
  tp.dq = static_cast<__nv_bfloat16*>(a->dq);
  tp.dk = static_cast<__nv_bfloat16*>(a->dk);
  tp.dv = static_cast<__nv_bfloat16*>(a->dv);
  tp.dbeta = static_cast<__nv_bfloat16*>(a->dbeta);
  tp.dg = a->dg;
  tp.g = a->g;
  if (P.gate) {
    tp.gate_act = 1;
    tp.lower_bound = d->lower_bound;
    tp.A_log = a->A_log;
    tp.dt_bias = a->dt_bias;
    tp.dA_part = R(L.dA_part);
    tp.ddt_part = R(L.ddt_part);
  }
  tp.status = a->status;
  tp.kda = kda ? 1 : 0;
  tp.sms = fp.sms;
  tp.qk_group = P.G;
  if (P.G > 1) {
    tp.dq32 = R(L.dq32);
    tp.dk32 = R(L.dk32);
  }

  {
    HeadGroups groups(P, true, s);
    for (int g = 0; g < groups.count(); ++g) {
      const cudaStream_t sg = groups.stream(g);
      pp.hg0 = cp.hg0 = rp.hg0 = fp.hg0 = tp.hg0 = groups.first(g);
      pp.hgn = cp.hgn = rp.hgn = fp.hgn = tp.hgn = groups.heads(g);
      if (!have_saved) {
        {
          TimedLaunch tl_(kKPrep, sg);
          rc = check_cuda(kda ? launch_prep_kda(M.q, M.k, M.v, pp, sg)
                              : launch_prep_gdn(M.q, M.k, M.v, M.Qt, M.Kt, M.Aqk, M.W, M.Usw, pp, sg),
                          "prepare kernel");
        }
        if (rc) return rc;
        rc = run_chain_fwd(P, M, cp, sg);
        if (rc) return rc;
      }
      rc = run_chain_bwd(P, M, rp, sg);
      if (rc) return rc;
      {
        TimedLaunch tl_(kKBwdFeat, sg);
        rc = check_cuda(launch_bwd_feat(M.VN, M.DVN, M.dO, M.Hs, M.DHs, fp, sg), "feature-major backward kernel");
      }
      if (rc) return rc;
      {
        TimedLaunch tl_(kKBwdTok, sg);
        rc = check_cuda(kda ? launch_bwd_tok_kda(M.q, M.k, M.v, M.VN, M.DW, M.DVN, M.dO, tp, sg)
                            : launch_bwd_tok(M.q, M.k, M.v, M.dO, M.VN, M.DW, M.DVN, tp, sg),
                        "token-major backward kernel");
      }
      if (rc) return rc;
    }
    rc = groups.join();
  }
  if (rc) return rc;
  if (P.gate) {
    GateGradParams gg{};
    gg.dA_part = tp.dA_part;
    gg.ddt_part = tp.ddt_part;
    gg.dA_log = a->dA_log;
    gg.ddt_bias = a->ddt_bias;
    gg.NC = P.NC;
    gg.H = P.H;
    TimedLaunch tl_(kKGateGrad, s);
    rc = check_cuda(launch_gate_grad(gg, s), "gate gradient kernel");
    if (rc) return rc;
  }
  if (P.G == 1) return GDN_OK;
  GroupSumParams gp{};
  gp.dq32 = tp.dq32;
  gp.dk32 = tp.dk32;
  gp.dq = tp.dq;
  gp.dk = tp.dk;
  gp.R = P.R;
  gp.H = P.H;
  gp.G = P.G;
  gp.sms = fp.sms;
  TimedLaunch tl_(kKGroupSum, s);
  return check_cuda(launch_group_sum(gp, s), "group sum kernel");
}

}  // namespace

// Records `msg` as the calling thread's last error (for entry points defined in other files).
int set_last_error(int code, const char* msg) { return fail(code, msg); }

// Timing hook brackets for launches made in other files (no-ops while timing is off).
TimedScope::TimedScope(int kind, cudaStream_t s) : impl_(new TimedLaunch(kind, s)) {}
TimedScope::~TimedScope() { delete static_cast<TimedLaunch*>(impl_); }

// Copies host offsets into device memory through kernel parameters (no staging buffer).
int upload_offsets(const int32_t* host, int count, int* dst, cudaStream_t s) {
  for (int off = 0; off < count; off += kMaxUploadInts) {
    UploadParams up;
    up.count = std::min(kMaxUploadInts, count - off);
    for (int i = 0; i < up.count; ++i) up.vals[i] = host[off + i];
    int rc = check_cuda(launch_upload(up, dst + off, s), "upload offsets");
    if (rc) return rc;
  }
  return GDN_OK;
}

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
    case GDN_ERANGE: return "per-channel gate outside the supported range";
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
  return make_layout(P, false).saved_total;
}

size_t gdn_saved_size(const gdn_desc_t* desc) {
  Problem P;
  if (validate_desc(desc, &P)) return 0;
  return make_layout(P, true, false).saved_total;
}

size_t kda_saved_size(const gdn_desc_t* desc) {
  Problem P;
  if (validate_desc(desc, &P)) return 0;
  return make_layout(P, true, true).saved_total;
}

size_t kda_fwd_workspace_size(const gdn_desc_t* desc) { return gdn_fwd_workspace_size(desc); }

size_t gdn_bwd_workspace_size(const gdn_desc_t* desc) {
  Problem P;
  if (validate_desc(desc, &P)) return 0;
  return make_layout(P, true).total;
}

size_t kda_bwd_workspace_size(const gdn_desc_t* desc) {
  Problem P;
  if (validate_desc(desc, &P)) return 0;
  return make_layout(P, true, true).total;
}

int gdn_set_chain_segment(int chunks) {
  if (chunks < 0) return fail(GDN_EINVAL, "segment length must be >= 0");
  g_chain_segment = chunks;
  return GDN_OK;
}

int gdn_set_head_groups(int groups) {
  if (groups < 0 || groups > 2) return fail(GDN_EINVAL, "head groups must be 0 (automatic), 1 or 2");
  g_head_groups = groups;
  return GDN_OK;
}

int gdn_chain_plan(const gdn_desc_t* desc, int* chunks_per_segment, int* max_segments) {
  Problem P;
  int rc = validate_desc(desc, &P);
  if (rc) return rc;
  if (!chunks_per_segment || !max_segments) return fail(GDN_EINVAL, "NULL output pointer");
  const ScanPlan sc = plan_scan(P);
  *chunks_per_segment = sc.L;
  *max_segments = sc.maxS;
  return GDN_OK;
}

int gdn_timing_enable(int enable) {
  g_tim.on = enable != 0;
  for (int k = 0; k < kKinds; ++k) g_tim.used[k] = 0;
  return GDN_OK;
}

int gdn_timing_kinds(void) { return kKinds; }

const char* gdn_timing_name(int kind) { return (kind >= 0 && kind < kKinds) ? kKindNames[kind] : ""; }

int gdn_timing_read(int kind, double* total_ms, int* launches) {
  if (kind < 0 || kind >= kKinds || !total_ms || !launches) return fail(GDN_EINVAL, "bad timing query");
  double tot = 0.0;
  for (size_t i = 0; i < g_tim.used[kind]; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(g_tim.ev[kind][i].second) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_tim.ev[kind][i].first, g_tim.ev[kind][i].second) != cudaSuccess)
      return fail(GDN_ECUDA, "timing event query failed");
    tot += ms;
  }
  *total_ms = tot;
  *launches = int(g_tim.used[kind]);
  g_tim.used[kind] = 0;
  return GDN_OK;
}

int gdn_fwd(const gdn_desc_t* desc, const gdn_fwd_args_t* args, void* stream) {
  g_err.clear();
  return run_fwd(desc, args, stream, false);
}

int kda_fwd(const gdn_desc_t* desc, const gdn_fwd_args_t* args, void* stream) {
  g_err.clear();
  return run_fwd(desc, args, stream, true);
}

int gdn_bwd(const gdn_desc_t* desc, const gdn_bwd_args_t* args, void* stream) {
  g_err.clear();
  return run_bwd(desc, args, stream, false);
}

int kda_bwd(const gdn_desc_t* desc, const gdn_bwd_args_t* args, void* stream) {
  g_err.clear();
  return run_bwd(desc, args, stream, true);
}

}  // extern "C"
