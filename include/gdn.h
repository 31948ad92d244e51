/* C ABI of libgdn: the chunkwise gated delta rule on one NVIDIA GB300 (sm_103a).
 *
 * Operations (forward and backward of one layer's recurrence):
 *   gdn_fwd / gdn_bwd : Gated DeltaNet, one scalar log-decay g per token and head.
 *   kda_fwd / kda_bwd : Kimi Delta Attention, one log-decay per token, head and key channel.
 *
 * What is computed. For every independent sequence (a dense batch row, or one document of a
 * packed row) and head, starting from S = initial_state (or 0), with K x V state S:
 *   qh = q / sqrt(|q|^2 + 1e-6), kh likewise        (when use_qk_l2norm; else qh = q, kh = k)
 *   b  = sigmoid(beta) when use_beta_sigmoid, else beta
 *   S' = exp(g_t) S           (GDN)   |   S' = diag(exp(g_t[:])) S   (KDA, per key channel)
 *   S  = S' + kh (b (v_t - S'^T kh))^T
 *   o_t = scale * S^T qh
 * This is the recurrence carried by the chunk loop of the eager reference
 * `torch_chunk_gated_delta_rule` (hyper-parallel GDN module, Diff Coverage page: `_l2norm`
 * with eps 1e-6 inside the square root, the cumulative-gate decay mask, the KK^T strictly
 * lower matrix and its forward-substitution inverse, the WY terms `value`/`k_cumdecay`, and
 * the per-chunk state update); the KDA form is the same rule with the per-channel
 * cumulative gate of the KDA staged native interface (`_KDAPrepared.gk`,
 * kimi_delta_attention_ascendc.py coverage page). The library evaluates it chunkwise with
 * 64-token chunks; results equal the recurrence up to rounding.
 *
 * Layout. Token-major BSND, contiguous: q, k [B,T,H,K]; v, o [B,T,H,V]; beta [B,T,H]; GDN g
 * [B,T,H]; KDA g [B,T,H,K]. States are [N,H,K,V] fp32 with N = B (dense) or the number of
 * documents (packed). K == V == 128. Packed documents use B == 1 and a HOST array
 * cu_seqlens of N+1 int32 offsets, 0 = c_0 < c_1 < ... < c_N = T; each document starts from
 * its own initial state and yields its own final state.
 *
 * Dtypes. q, k, v, o, beta, dq, dk, dv, dbeta, dO: bf16 (passed as uint16 bit patterns).
 * g, dg, states, dht, dh0: fp32. Arithmetic: fp32 accumulation; tensor-core operands bf16
 * where they are exact input values, tf32 (round-to-nearest) elsewhere, except the per-chunk
 * copies of the state and of its gradient that the backward's feature-major products read,
 * which are kept in bf16 (round-to-nearest).
 *
 * Ownership. Every pointer in the argument structs is a DEVICE pointer owned by the caller,
 * except cu_seqlens (HOST). The library never allocates or frees memory: the caller passes a
 * device workspace of at least *_workspace_size() bytes (256-byte aligned). q, k, v, o (and
 * dO, dq, dk, dv in the backward) must be 16-byte aligned (tensor-memory-access copies and
 * vector stores).
 * No output may alias an input. cu_seqlens is read during the call only.
 *
 * Asynchrony and errors. Validation is host-side and synchronous; on success the work is
 * enqueued on `stream` (a cudaStream_t, NULL = legacy default stream) and the call returns
 * GDN_OK without synchronising. A contract violation returns GDN_EINVAL before anything is
 * enqueued (gdn_last_error() gives the reason); a device other than compute capability 10.3
 * gives GDN_EUNSUPPORTED; a CUDA launch failure gives GDN_ECUDA. Device kernels never trap:
 * every wait inside a kernel is bounded and, when it runs out, records a nonzero code in the
 * caller's `status` word (an int in device memory, or NULL), which the caller may read after
 * synchronising: 1, 2 or 3 (a TMA, MMA or thread wait ran out: GDN_ETIMEOUT semantics) or
 * GDN_ERANGE (below). The first code recorded stays; every entry point that starts from the
 * inputs resets the word to 0.
 *
 * Gate range. GDN: any g <= 0 is accepted; g is floored at -128 inside the kernels, where
 * exp(g) is already 0 in fp32, so g = -inf (or any g <= -128) is an exact state reset and dg
 * there is 0. KDA: within every 16-token block of a chunk (tokens 16i .. 16i+15 of the chunk),
 * each channel's cumulative gate may change by at most 80 from its value at the block's first
 * token. This covers the pages' safe-gate range (every g in [-5, 0]: at most 75). A call outside
 * it records GDN_ERANGE in the status word and its results are undefined.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_OK 0
#define GDN_EINVAL 1        /* contract violation: shapes, flags, offsets, pointers, workspace */
#define GDN_EUNSUPPORTED 2  /* not a compute-capability 10.3 device, or no device */
#define GDN_ECUDA 3         /* a CUDA runtime call or kernel launch failed */
#define GDN_ETIMEOUT 4      /* a bounded in-kernel wait ran out (reported via the status word) */
#define GDN_ERANGE 5        /* a KDA gate outside the supported range (reported via the status word) */

/* Problem description shared by every entry point. */
typedef struct {
  int B, T, H, K, V;         /* dense: B >= 1; packed (cu_seqlens != NULL): B == 1. K == V == 128 */
  int chunk_size;            /* must be 64 */
  const int32_t* cu_seqlens; /* HOST, num_seqs + 1 offsets, or NULL for dense */
  int num_seqs;              /* documents when packed; ignored (== B) when dense */
  float scale;               /* output scale; <= 0 selects 1/sqrt(K) */
  int use_qk_l2norm;         /* L2-normalise q and k per token and head (eps 1e-6) */
  int use_beta_sigmoid;      /* beta holds logits; the kernel applies sigmoid */
  int output_final_state;    /* write final_state */
  int num_k_heads;           /* heads of q and k (grouped-query layout: H value heads share them,
                                value head h reads q/k head h / (H / num_k_heads), the pages'
                                `repeat_interleave` of q and k, done by indexing); must divide H;
                                0 means H. dq and dk are the sums over each group. */
  int use_gate_in_kernel;    /* KDA only (0 for GDN): g holds gate logits x and the kernels use the
                                activated gate lower_bound * sigmoid(exp(A_log[h]) (x + dt_bias[h][k]))
                                (the KDA page's `_prepare_kda` with use_gate_in_kernel and safe_gate;
                                the formula is this library's reading: the pages give the interface,
                                the range and the gradients, not the expression) */
  float lower_bound;         /* the safe gate's bound, in [-5, 0) (used with use_gate_in_kernel) */
} gdn_desc_t;

typedef struct {
  const void* q;             /* bf16 [B,T,Hk,K] (Hk = num_k_heads, or H) */
  const void* k;             /* bf16 [B,T,Hk,K] */
  const void* v;             /* bf16 [B,T,H,V] */
  const float* g;            /* GDN [B,T,H], KDA [B,T,H,K]: natural-log decay, <= 0 expected */
  const void* beta;          /* bf16 [B,T,H] */
  const float* initial_state;/* [N,H,K,V] or NULL (zeros) */
  void* o;                   /* bf16 [B,T,H,V], written */
  float* final_state;        /* [N,H,K,V], written when output_final_state (else may be NULL) */
  void* workspace;           /* device, >= *_fwd_workspace_size() bytes, 256-byte aligned
                                (ignored, may be NULL, when `saved` is given) */
  size_t workspace_bytes;
  int* status;               /* device int or NULL: nonzero after a bounded wait ran out */
  void* saved;               /* training: device buffer of >= *_saved_size() bytes (256-byte
                                aligned) that receives the chunk intermediates the backward
                                needs; NULL for inference */
  size_t saved_bytes;
  const float* A_log;        /* use_gate_in_kernel: [H] fp32 (else ignored) */
  const float* dt_bias;      /* use_gate_in_kernel: [H,K] fp32 (else ignored) */
} gdn_fwd_args_t;

typedef struct {
  const void* q;             /* forward inputs, as passed to the forward */
  const void* k;
  const void* v;
  const float* g;
  const void* beta;
  const float* initial_state;/* [N,H,K,V] or NULL */
  const void* dO;            /* bf16 [B,T,H,V]: gradient of the output */
  const float* dht;          /* [N,H,K,V] gradient of the final state, or NULL */
  void* dq;                  /* bf16 [B,T,Hk,K] (summed over each group of value heads) */
  void* dk;                  /* bf16 [B,T,Hk,K] */
  void* dv;                  /* bf16 [B,T,H,V] */
  void* dbeta;               /* bf16 [B,T,H]: w.r.t. beta as passed (the logit when use_beta_sigmoid) */
  float* dg;                 /* fp32, same shape as g: w.r.t. the raw per-token gate */
  float* dh0;                /* [N,H,K,V] or NULL */
  void* workspace;           /* >= *_bwd_workspace_size() bytes; with `saved`, >= that minus
                                *_saved_size() bytes */
  size_t workspace_bytes;
  int* status;
  const void* saved;         /* the `saved` buffer of a forward with the same description and
                                inputs (the backward then skips recomputing the forward), or
                                NULL (the backward recomputes it) */
  size_t saved_bytes;
  const float* A_log;        /* use_gate_in_kernel: the forward's gate parameters */
  const float* dt_bias;
  float* dA_log;             /* use_gate_in_kernel: [H] fp32, written (else ignored). dg is then the
                                gradient w.r.t. the gate logits x */
  float* ddt_bias;           /* use_gate_in_kernel: [H,K] fp32, written */
} gdn_bwd_args_t;

/* Human-readable name of an error code. */
const char* gdn_strerror(int code);
/* Reason for the last GDN_EINVAL / GDN_ECUDA returned on the calling thread ("" if none). */
const char* gdn_last_error(void);
/* GDN_OK if `device` is a compute-capability 10.3 GPU this library was built for. */
int gdn_device_supported(int device);

/* Workspace sizes in bytes for a valid description; 0 when the description is invalid. */
size_t gdn_fwd_workspace_size(const gdn_desc_t* desc);
size_t gdn_bwd_workspace_size(const gdn_desc_t* desc);
size_t kda_fwd_workspace_size(const gdn_desc_t* desc);
size_t kda_bwd_workspace_size(const gdn_desc_t* desc);
/* Size of the optional saved-intermediates buffer a training forward fills for its backward
 * (the save mode of the pages' native interfaces; recompute when it is not used). */
size_t gdn_saved_size(const gdn_desc_t* desc);
size_t kda_saved_size(const gdn_desc_t* desc);

/* Gated DeltaNet forward: o (and final_state). */
int gdn_fwd(const gdn_desc_t* desc, const gdn_fwd_args_t* args, void* stream);
/* Gated DeltaNet backward: gradients of <dO, o> + <dht, final_state> w.r.t. q, k, v, beta,
 * g and initial_state (dh0). The forward's intermediates come from `saved`, or are
 * recomputed from the inputs when `saved` is NULL. */
int gdn_bwd(const gdn_desc_t* desc, const gdn_bwd_args_t* args, void* stream);
/* Kimi Delta Attention forward / backward: as above with the per-channel gate g [B,T,H,K]. */
int kda_fwd(const gdn_desc_t* desc, const gdn_fwd_args_t* args, void* stream);
int kda_bwd(const gdn_desc_t* desc, const gdn_bwd_args_t* args, void* stream);

/* Allocation-free forward (no counterpart in the paper: an interface addition for callers
 * that cannot allocate device memory when they run the layer, such as code inside a CUDA
 * graph capture, embedders bound to a framework allocator, or latency-critical paths).
 * Same computation and arguments as gdn_fwd, except that args->workspace and args->saved
 * must be NULL and their sizes 0: the workspace is a fixed static device array of
 * gdn_fwd_noalloc_capacity() bytes (32 MiB) inside this library, held by every GPU that loads
 * it until exit. Problems whose gdn_fwd_workspace_size() exceeds it return GDN_EINVAL. The call
 * itself allocates nothing. All calls on a device share that array (it keeps the last call's
 * contents; nothing needs clearing), so calls that overlap on the GPU race and must not be
 * issued. The first call on each device, with that device current, looks the array's device
 * address up once; make it before any stream capture. */
int gdn_fwd_noalloc(const gdn_desc_t* desc, const gdn_fwd_args_t* args, void* stream);
size_t gdn_fwd_noalloc_capacity(void);

/* Segmented state chain (no counterpart in the paper's kernels; it runs the pages' affine
 * state summary, state_out = M state_in + S and its adjoint, inside one GPU instead of across
 * context-parallel ranks: hyper-parallel GDN Diff Coverage page,
 * `_compute_gdn_state_summary_from_prepared` / `_apply_gdn_state_summary`). The serial
 * inter-chunk recurrence of each (sequence, head) is cut into segments of L chunks; the
 * segments' affine maps are computed in parallel, composed, and the segments rerun from their
 * entry states. The result equals the plain chain up to rounding. L is chosen per call from
 * the problem's shape (gdn_chain_plan() reports the choice: L and the largest number of
 * segments of any sequence; 1 segment = the plain chain). gdn_set_chain_segment(L) forces L
 * for every later call and size query of the process (0 restores the automatic choice; a
 * value at least the longest sequence's chunk count selects the plain chain); the workspace
 * and saved sizes depend on it, so it must not change between a size query and the calls
 * that use the buffers. Process-global, not thread-safe. Negative L: GDN_EINVAL. */
int gdn_set_chain_segment(int chunks);
int gdn_chain_plan(const gdn_desc_t* desc, int* chunks_per_segment, int* max_segments);

/* Head groups (no counterpart in the paper; a scheduling choice of this library). A problem
 * with at least 8 heads and enough chunk-heads (chunks of all sequences x heads: 1024 for a
 * backward, 4096 for a forward) splits its heads into two groups: the first group's
 * kernels run on the caller's stream, the second group's on a stream that the library creates
 * once per device, forked after the work already enqueued on the caller's stream and joined
 * back into it before the call returns, so ordering on the caller's stream is unchanged. The
 * two groups then share the GPU, and one group's low-occupancy phases overlap the other's work.
 * Results are identical with and without the split (every head is computed independently).
 * gdn_set_head_groups(n) forces n groups (1 or 2) for every later call of the process; 0
 * restores the automatic choice. Process-global, not thread-safe; other values: GDN_EINVAL. */
int gdn_set_head_groups(int groups);

/* Short convolution ahead of the path: causal depthwise Conv1d over the token axis with
 * optional bias and SiLU, per packed document (hyper-parallel GDN Diff Coverage page,
 * `_causal_conv1d_with_cp_halo` and the packed ShortConv path, which produce q, k and v):
 *   z[t][c] = bias[c] + sum_{i<W} weight[c][i] x[t - (W-1-i) dilation][c],  y = silu(z) or z.
 * Positions before a sequence's first token read that sequence's halo (its (W-1) dilation
 * preceding tokens, e.g. another context-parallel rank's tail) or zero. Rows never read
 * across packed-document boundaries. */
typedef struct {
  int B, T, C;               /* x is [B,T,C]; packed (cu_seqlens != NULL): B == 1. C % 8 == 0 */
  int W;                     /* taps, 1..8 */
  int dilation;              /* >= 1 */
  const int32_t* cu_seqlens; /* HOST, num_seqs + 1 offsets, or NULL for dense */
  int num_seqs;
  int activation;            /* 1: SiLU, 0: none */
} gdn_conv_desc_t;

typedef struct {
  const void* x;             /* bf16 [B,T,C], 16-byte aligned */
  const float* weight;       /* fp32 [C,W], 16-byte aligned */
  const float* bias;         /* fp32 [C] or NULL, 16-byte aligned */
  const void* halo;          /* bf16 [N,(W-1)*dilation,C] or NULL (zeros) */
  void* y;                   /* bf16 [B,T,C], 16-byte aligned, written */
  void* workspace;           /* >= gdn_conv_fwd_workspace_size() bytes, 256-byte aligned */
  size_t workspace_bytes;
} gdn_conv_fwd_args_t;

typedef struct {
  const void* x;             /* forward inputs, as passed to the forward */
  const float* weight;
  const float* bias;
  const void* halo;
  const void* dy;            /* bf16 [B,T,C] gradient of y */
  void* dx;                  /* bf16 [B,T,C], written */
  float* dweight;            /* fp32 [C,W], written */
  float* dbias;              /* fp32 [C], written, or NULL */
  float* dhalo;              /* fp32 [N,(W-1)*dilation,C], written, or NULL */
  void* workspace;           /* >= gdn_conv_bwd_workspace_size() bytes, 256-byte aligned */
  size_t workspace_bytes;
} gdn_conv_bwd_args_t;

size_t gdn_conv_fwd_workspace_size(const gdn_conv_desc_t* desc);
size_t gdn_conv_bwd_workspace_size(const gdn_conv_desc_t* desc);
int gdn_conv_fwd(const gdn_conv_desc_t* desc, const gdn_conv_fwd_args_t* args, void* stream);
int gdn_conv_bwd(const gdn_conv_desc_t* desc, const gdn_conv_bwd_args_t* args, void* stream);

/* Profiling hooks (not part of the computation). While enabled, every kernel launch of the
 * calls above is bracketed by CUDA events on its stream. gdn_timing_read() synchronizes the
 * recorded events of one kernel kind (0 .. gdn_timing_kinds()-1, named by gdn_timing_name()),
 * returns their summed device time in milliseconds and the number of launches, and clears
 * them. Process-global state, not thread-safe; enabling resets all counters. */
int gdn_timing_enable(int enable);
int gdn_timing_kinds(void);
const char* gdn_timing_name(int kind);
int gdn_timing_read(int kind, double* total_ms, int* launches);

/* Self-test of the failure reporting of the bounded in-kernel waits (no counterpart in the
 * pages: a check of this library's own error path, not part of the computation). Enqueues one
 * small kernel on `stream` whose threads wait, with a limit of `limit_ns` nanoseconds
 * (0 < limit_ns <= 2e9), on a barrier that nothing completes, while one 4096-byte copy from
 * `src` (device, 16-byte aligned, at least 4096 bytes, only read) is in flight. The wait runs
 * out, records 3 (a thread wait ran out: GDN_ETIMEOUT semantics) in the device int `*status`
 * (which the caller zeroes beforehand) and the kernel exits normally after the copy has landed;
 * the stream and the context stay usable. Returns GDN_EINVAL for bad arguments, GDN_EUNSUPPORTED
 * off compute capability 10.3, else GDN_OK without synchronising. */
int gdn_wait_selftest(const void* src, long long limit_ns, int* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_H */
