// Shared definitions of the gated-delta-rule kernels: chunk tables, workspace tiles and the
// parameter blocks the host passes to each kernel.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace gdn {

constexpr int kC = 64;     // chunk length (tokens)
constexpr int kD = 128;    // head dim K == V
constexpr int kMaxUploadInts = 4000;  // cu_seqlens entries per upload launch

// One chunk of one sequence: {first token row (flattened B*T), valid rows (1..64),
// sequence index, chunk index within the sequence}.
using ChunkEntry = int4;
// One sequence: {first chunk index, number of chunks}.
using SeqEntry = int2;

// Per-(chunk, head) workspace tiles written by the prepare kernel (fp32):
//   W   [64][128]  A diag(beta exp(G) r_k) k        (k_cumdecay; state feedback)
//   U   [64][128]  A diag(beta) v                    (chunk value)
//   Qt  [64][128]  scale r_q exp(G) q               (gated, scaled queries)
//   KtT [128][64]  (r_k exp(G_last - G) k)^T        (keys decayed to the chunk end)
//   Aqk [64][64]   scale r_q r_k (q k^T) exp(G_i - G_j), i >= j
//   gam [128]      exp(G_last) (per key channel; GDN fills entry 0 only)
constexpr size_t kTileW = size_t(kC) * kD;
constexpr size_t kTileKtT = size_t(kD) * kC;
constexpr size_t kTileAqk = size_t(kC) * kC;

struct PrepParams {
  const ChunkEntry* chunks;
  int NC, H;
  const float* g;              // GDN [R,H]; KDA [R,H,K]
  const __nv_bfloat16* beta;   // [R,H]
  float scale;
  int l2norm, beta_sigmoid;
  float *W, *U, *Qt, *KtT, *Aqk, *gam;
  float *Gc, *rq, *rk, *beff;  // optional per-token saves [NC*H*64] (KDA Gc: [NC*H*64*128]); may be null
  // Backward-only tiles (all null in the forward):
  float* Kt;                   // [64][128]  r_k exp(G_last - G) k   (row-major KtT^T)
  float* QtT;                  // [128][64]  Qt^T
  float* AqkT;                 // [64][64]   Aqk^T
  float* WT;                   // [128][64]  W^T
  float* A;                    // [64][64]   (I + L)^-1
  int* status;
};

struct RevChainParams {
  const SeqEntry* seqs;
  const ChunkEntry* chunks;
  int N, H;
  int kda;
  const float* gam;            // [NC,H,128]
  const __nv_bfloat16* dO;     // [R,H,V]
  const float* dht;            // [N,H,K,V] or null
  float* dh0;                  // [N,H,K,V] or null
  float* dh_save;              // [NC,H,K,V] gradient w.r.t. the state leaving each chunk
  float* dvn_save;             // [NC,H,64,V] gradient w.r.t. v_new
  int* status;
};

struct ChainParams {
  const SeqEntry* seqs;
  const ChunkEntry* chunks;
  int N, H;
  int kda;
  const float* gam;
  const float* h0;             // [N,H,K,V] or null
  float* hT;                   // [N,H,K,V] or null
  __nv_bfloat16* o;            // [R,H,V] or null
  float* h_save;               // [NC,H,K,V] entry state of every chunk, or null
  float* vnew_save;            // [NC,H,64,V] or null
  int* status;
};

struct TableParams {
  const int* cu;               // device copy of cu_seqlens (N+1) or null for dense
  int N, T, NC;
  SeqEntry* seqs;
  ChunkEntry* chunks;
  int* status;                 // caller's status word, reset to 0 here (may be null)
};

struct UploadParams {
  int count;
  int vals[kMaxUploadInts];
};

struct BwdFeatParams {
  const ChunkEntry* chunks;
  int NC, H, kda;
  const float* h;              // [NC,H,K,V] state entering each chunk
  const float* dh;             // [NC,H,K,V] gradient w.r.t. the state leaving each chunk
  const __nv_bfloat16* dO;     // [R,H,V]
  const float* A;              // [NC,H,64,64]
  const float* dvn;            // [NC,H,64,V]
  float *dQt, *dKt, *dW, *dK1, *dV1;  // [NC,H,64,128] token-major
  float* dgam;                 // [NC,H,128] (GDN: entry 0)
  int* status;
};

struct BwdTokParams {
  const ChunkEntry* chunks;
  int NC, H, kda;
  float scale;
  int beta_sigmoid, l2norm;
  const __nv_bfloat16* dO;     // [R,H,V]
  const float* A;              // [NC,H,64,64]
  const float *Gc, *rq, *rk, *beff;   // per token [NC,H,64]
  const float *dQt, *dKt, *dK1, *dV1; // [NC,H,64,128]
  const float *gam, *dgam;     // [NC,H,128]
  __nv_bfloat16 *dq, *dk, *dv, *dbeta;
  float* dg;
  int* status;
};

// Launchers (defined next to their kernels). Return the cudaError_t of the launch.
cudaError_t launch_upload(const UploadParams& p, int* dst, cudaStream_t s);
cudaError_t launch_tables(const TableParams& p, cudaStream_t s);
cudaError_t launch_prep_gdn(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const PrepParams& p, cudaStream_t s);
cudaError_t launch_prep_kda(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const PrepParams& p, cudaStream_t s);
cudaError_t launch_chain_bwd(const CUtensorMap& mKt, const CUtensorMap& mAqkT, const CUtensorMap& mQtT,
                             const CUtensorMap& mWT, const RevChainParams& p, cudaStream_t s);
cudaError_t launch_bwd_feat(const CUtensorMap& mVN, const CUtensorMap& mDVN, const BwdFeatParams& p, cudaStream_t s);
cudaError_t launch_bwd_tok(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mVN,
                           const CUtensorMap& mDW, const CUtensorMap& mDVN, const BwdTokParams& p, cudaStream_t s);
cudaError_t launch_bwd_tok_kda(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                               const CUtensorMap& mVN, const CUtensorMap& mDW, const CUtensorMap& mDVN,
                               const BwdTokParams& p, cudaStream_t s);
cudaError_t launch_chain_fwd(const CUtensorMap& mW, const CUtensorMap& mQt, const CUtensorMap& mKtT,
                             const CUtensorMap& mAqk, const CUtensorMap& mU, const ChainParams& p,
                             cudaStream_t s);

}  // namespace gdn
