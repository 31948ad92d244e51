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
constexpr float kLog2e = 1.4426950408889634f;  // log2(e): exp(x) = exp2(x log2(e))
// Floor on the scalar per-token log-decay g of Gated DeltaNet. exp(-128) is below the smallest
// fp32 subnormal after the log2 scaling (2^-184.7), so every decay factor that spans a floored
// token is exactly 0 in fp32, which is what exp(g) gives for g = -inf (a hard state reset).
// Flooring keeps the chunk-local cumulative gate finite, so differences G_i - G_j of two
// positions after a reset stay exact sums instead of (-inf) - (-inf).
constexpr float kGateFloor = -128.f;
// Largest drop of a per-channel cumulative gate (natural log) within one 16-token block that
// the per-channel prepare kernel accepts: its block factorisation splits exp(G_i - G_j) into
// exp(G_i - G_r) exp(G_r - G_j) around the block's first row r, and both factors stay normal
// fp32 numbers while the drop is at most 80 (exp(-80) = 1.8e-35). Gates in the pages'
// safe-gate range [-5, 0] drop at most 75 over 15 tokens.
constexpr float kKdaBlockDropMax = 80.f;

// One chunk of one sequence: {first token row (flattened B*T), valid rows (1..64),
// sequence index, chunk index within the sequence}.
using ChunkEntry = int4;

// Chunk c's table entry {first row, rows, sequence, chunk within the sequence}: computed for a
// dense batch (every sequence dense_T tokens, chunks numbered sequence by sequence), so a CTA
// can issue its first copies without waiting for the table; loaded for packed documents.
__device__ __forceinline__ ChunkEntry chunk_entry(const ChunkEntry* chunks, int c, int dense_T) {
  if (dense_T > 0) {
    const int ncs = (dense_T + kC - 1) / kC, n = c / ncs, j = c - n * ncs;
    return make_int4(n * dense_T + j * kC, min(kC, dense_T - j * kC), n, j);
  }
  return chunks[c];
}
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

// Writes a thread's N fp32 values s[e] as bf16 into column v, rows 0..N-1, of a row-major
// [rows][kD] bf16 tile at `base` (the chain kernels' state saves and the feature-major backward's
// token-major results, where lane v holds column v). Lanes v and v ^ 1 (same warp, same rows)
// swap one value per row pair, so each store writes two adjacent columns: the even lane the even
// rows, the odd lane the odd rows. Every lane of the warp must take part.
template <int N>
__device__ __forceinline__ void store_col_bf16(__nv_bfloat16* base, const float* s, int v) {
  const int odd = v & 1;
  __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(base + (v & ~1));
#pragma unroll
  for (int e = 0; e < N; e += 2) {
    const float other = __shfl_xor_sync(0xffffffffu, odd ? s[e] : s[e + 1], 1);
    const __nv_bfloat162 pr = odd ? __floats2bfloat162_rn(other, s[e + 1]) : __floats2bfloat162_rn(s[e], other);
    p[size_t(e + odd) * (kD / 2)] = pr;
  }
}

// Four consecutive bf16 (8 bytes, 8-byte aligned) of read-only memory as fp32.
__device__ __forceinline__ float4 ldg_bf16x4(const __nv_bfloat16* src) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(src));
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

// Segmented chain (chunk-parallel affine state scan). The chunk map of the chain is affine
// in the state, S_out = M_c S_in + B_c with M_c = diag(gam) - k~^T W and B_c = k~^T U
// (the affine state summary of the pages' context-parallel GDN path, composed over chunks);
// the reverse chain's map is its adjoint. Each sequence's chunks are cut into segments of L
// chunks (the last may be shorter), numbered in processing order (reverse chain: from the
// sequence's end). Pass 0 runs segment 0 in full from the true initial state and, for every
// segment 1..ns-2, the segment's map twice: from the identity with no input (giving M) and
// from zero with the input (giving B). A compose kernel then walks the segments, E[s+1] =
// M_s E[s] + B_s, and pass 1 runs segments 1..ns-1 in full from E[s]. L >= every sequence's
// chunk count (maxS == 1) is the plain serial chain.
enum RunMode : int { kRunFull = 0, kRunMapM = 1, kRunMapB = 2 };

// Grids: the chain kernels launch (runs, heads of the group); the chunk kernels (prepare and
// the two backward kernels) launch one flat dimension of chunk x heads with the head fastest,
// so the CTAs in flight read whole token rows of the [T, H, 128] inputs and neighbouring
// per-(chunk, head) tiles.

struct SegPlan {
  int L;       // chunks per segment
  int maxS;    // most segments of any sequence (1 = plain chain)
  int pass;    // 0 or 1
  float* E;    // [N*maxS*H][128][128] entry state (reverse: exit gradient) of each segment
  float* Phi;  // [N*maxS*H][128][128] segment map M, transposed (row j = column j of M), fp32
  float* Bm;   // [N*maxS*H][128][128] segment offset B
};

// CTAs per sequence (and head) of a chain pass.
__host__ __device__ inline int runs_per_seq(int maxS, int pass) {
  return pass == 0 ? (maxS <= 2 ? 1 : 2 * maxS - 3) : maxS - 1;
}

// Segment and mode of run `slot` of a pass for a sequence of `ns` segments; false when the
// sequence has no such run (the CTA exits at once).
__host__ __device__ inline bool decode_run(int slot, int pass, int ns, int* seg, int* mode) {
  if (pass == 0) {
    if (slot == 0) {
      *seg = 0;
      *mode = kRunFull;
      return true;
    }
    const int i = (slot - 1) >> 1;
    *seg = 1 + i;
    *mode = ((slot - 1) & 1) ? kRunMapB : kRunMapM;
    return 1 + i <= ns - 2;
  }
  *seg = 1 + slot;
  *mode = kRunFull;
  return 1 + slot <= ns - 1;
}

struct PrepParams {
  const ChunkEntry* chunks;
  int NC, H;
  int dense_T;                 // tokens per sequence of a dense batch (chunk entries computed), 0 if packed
  int hg0, hgn;                // head group: heads hg0 .. hg0 + hgn - 1
  const float* g;              // GDN [R,H]; KDA [R,H,K]
  const __nv_bfloat16* beta;   // [R,H]
  float scale;
  int l2norm, beta_sigmoid;
  int qk_group;                // value heads per q/k head (q/k head of value head h: h / qk_group)
  float *W, *U, *Qt, *KtT, *Aqk, *gam;
  float *Gc, *rq, *rk, *beff;  // optional per-token saves [NC*H*64] (KDA Gc: [NC*H*64*128]); may be null
  // Backward-only tiles (all null in the forward):
  float* Kt;                   // [64][128]  r_k exp(G_last - G) k   (row-major KtT^T)
  float* QtT;                  // [128][64]  Qt^T
  float* AqkT;                 // [64][64]   Aqk^T
  float* WT;                   // [128][64]  W^T
  float* A;                    // [64][64]   (I + L)^-1
  // In-kernel KDA gate activation: g holds logits x; the gate is
  // lower_bound * sigmoid(exp(A_log[h]) (x + dt_bias[h][k])).
  int gate_act;
  float lower_bound;
  const float* A_log;          // [H]
  const float* dt_bias;        // [H,K]
  int* status;
};

struct RevChainParams {
  const SeqEntry* seqs;
  const ChunkEntry* chunks;
  int N, H;
  int hg0, hgn;                // head group: heads hg0 .. hg0 + hgn - 1
  int kda;
  SegPlan sp;
  const float* gam;            // [NC,H,128]
  const __nv_bfloat16* dO;     // [R,H,V]
  const float* dht;            // [N,H,K,V] or null
  float* dh0;                  // [N,H,K,V] or null
  __nv_bfloat16* dh_save;      // [NC,H,K,V] gradient w.r.t. the state leaving each chunk (bf16)
  float* dvn_save;             // [NC,H,64,V] gradient w.r.t. v_new
  int* status;
};

struct ChainParams {
  const SeqEntry* seqs;
  const ChunkEntry* chunks;
  int N, H;
  int hg0, hgn;                // head group: heads hg0 .. hg0 + hgn - 1
  int kda;
  SegPlan sp;
  const float* gam;
  const float* h0;             // [N,H,K,V] or null
  float* hT;                   // [N,H,K,V] or null
  __nv_bfloat16* o;            // [R,H,V] or null
  __nv_bfloat16* h_save;       // [NC,H,K,V] entry state of every chunk (bf16), or null
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
  int dense_T;                 // tokens per sequence of a dense batch (chunk entries computed), 0 if packed
  int hg0, hgn;                // head group: heads hg0 .. hg0 + hgn - 1
  const __nv_bfloat16* h;      // [NC,H,K,V] state entering each chunk (bf16; read by TMA)
  const __nv_bfloat16* dh;     // [NC,H,K,V] gradient w.r.t. the state leaving each chunk (bf16; read by TMA)
  const __nv_bfloat16* dO;     // [R,H,V]
  const float* A;              // [NC,H,64,64]
  const float* dvn;            // [NC,H,64,V]
  __nv_bfloat16 *dQt, *dKt, *dK1;    // [NC,H,64,128] token-major, bf16
  float *dW, *dV1;                    // [NC,H,64,128] token-major
  float* dgam;                 // [NC,H,128] (GDN: entry 0)
  int sms;                     // SM count (the distance to the next wave's CTA for prefetching)
  int* status;
};

struct BwdTokParams {
  const ChunkEntry* chunks;
  int NC, H, kda;
  int dense_T;                 // tokens per sequence of a dense batch (chunk entries computed), 0 if packed
  int hg0, hgn;                // head group: heads hg0 .. hg0 + hgn - 1
  float scale;
  int beta_sigmoid, l2norm;
  const __nv_bfloat16* dO;     // [R,H,V]
  const float* A;              // [NC,H,64,64]
  const float *Gc, *rq, *rk, *beff;   // per token [NC,H,64]
  const __nv_bfloat16 *dQt, *dKt, *dK1;  // [NC,H,64,128] token-major, bf16
  const float* dV1;                      // [NC,H,64,128] token-major
  const float *gam, *dgam;     // [NC,H,128]
  __nv_bfloat16 *dq, *dk, *dv, *dbeta;
  float* dg;
  const float* g;              // the raw gate as passed ([R,H] GDN floor test; [R,H,K] KDA logits)
  int gate_act;                // KDA in-kernel gate activation (see PrepParams)
  float lower_bound;
  const float* A_log;
  const float* dt_bias;
  float *dA_part, *ddt_part;   // gate_act: per (chunk, head, channel) partial sums [NC,H,K]
  int qk_group;                // value heads per q/k head
  float *dq32, *dk32;          // qk_group > 1: per-value-head dq, dk [R,H,K] fp32 (summed later)
  int sms;                     // SM count (the distance to the next wave's CTA for prefetching)
  int* status;
};

// Kernel kinds of the per-launch timing hook (names in api.cu).
enum KernelKind {
  kKTables = 0, kKPrep, kKChainFwd, kKChainBwd, kKBwdFeat, kKBwdTok, kKCompose, kKGroupSum, kKConvFwd, kKConvBwd,
  kKGateGrad, kKinds
};

// Host helpers shared by the entry points of several files (api.cu).
int set_last_error(int code, const char* msg);
int upload_offsets(const int32_t* host, int count, int* dst, cudaStream_t s);
class TimedScope {  // records CUDA events around the launches in its scope while timing is on
 public:
  TimedScope(int kind, cudaStream_t s);
  ~TimedScope();
 private:
  void* impl_;
};

// Launchers (defined next to their kernels). Return the cudaError_t of the launch.
cudaError_t launch_upload(const UploadParams& p, int* dst, cudaStream_t s);
cudaError_t launch_tables(const TableParams& p, cudaStream_t s);
cudaError_t launch_prep_gdn(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const CUtensorMap& mQt, const CUtensorMap& mKt, const CUtensorMap& mAqk,
                            const CUtensorMap& mW, const CUtensorMap& mU, const PrepParams& p, cudaStream_t s);
cudaError_t launch_prep_kda(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const PrepParams& p, cudaStream_t s);
cudaError_t launch_chain_bwd(const CUtensorMap& mKt, const CUtensorMap& mAqkT, const CUtensorMap& mQtT,
                             const CUtensorMap& mWT, const CUtensorMap& mdO, const RevChainParams& p,
                             cudaStream_t s);
cudaError_t launch_bwd_feat(const CUtensorMap& mVN, const CUtensorMap& mDVN, const CUtensorMap& mdO,
                            const CUtensorMap& mH, const CUtensorMap& mDH, const BwdFeatParams& p, cudaStream_t s);
cudaError_t launch_bwd_tok(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdO,
                           const CUtensorMap& mVN, const CUtensorMap& mDW, const CUtensorMap& mDVN, const BwdTokParams& p,
                           cudaStream_t s);
cudaError_t launch_bwd_tok_kda(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                               const CUtensorMap& mVN, const CUtensorMap& mDW, const CUtensorMap& mDVN,
                               const CUtensorMap& mdO, const BwdTokParams& p, cudaStream_t s);
struct GroupSumParams {
  const float *dq32, *dk32;    // [R,H,K]
  __nv_bfloat16 *dq, *dk;      // [R,H/G,K]
  long long R;
  int H, G;
  int sms;                     // SM count of the device (grid size)
};

struct ComposeParams {
  const SeqEntry* seqs;
  int N, H;
  int hg0, hgn;                // head group: heads hg0 .. hg0 + hgn - 1
  SegPlan sp;
  int* status;
};

cudaError_t launch_group_sum(const GroupSumParams& p, cudaStream_t s);

// Gradients of the KDA gate parameters from the token-backward's per-chunk partial sums:
// ddt_bias[h][k] = sum over chunks of ddt_part, dA_log[h] = sum over chunks and channels of
// dA_part, in a fixed order (deterministic).
struct GateGradParams {
  const float *dA_part, *ddt_part;  // [NC,H,K]
  float *dA_log, *ddt_bias;         // [H], [H,K]
  int NC, H;
};
cudaError_t launch_gate_grad(const GateGradParams& p, cudaStream_t s);
cudaError_t launch_compose(const ComposeParams& p, cudaStream_t s);
cudaError_t launch_chain_fwd(const CUtensorMap& mW, const CUtensorMap& mQt, const CUtensorMap& mKtT,
                             const CUtensorMap& mAqk, const CUtensorMap& mU, const ChainParams& p,
                             cudaStream_t s);

}  // namespace gdn
