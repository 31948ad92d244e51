// Reverse chain kernel: the serial backward recurrence of the state gradient.
//
// For the forward chunk map  v_new = U - W S,  o = Qt S + Aqk v_new,
// S' = diag(gam) S + k~^T v_new  (k~ = Kt, keys decayed to the chunk end), the adjoint,
// with dS' the gradient w.r.t. the state leaving the chunk and dO the output gradient, is
//   dv_new = Aqk^T dO + Kt dS'
//   dS     = diag(gam) dS' + Qt^T dO - W^T dv_new
// run from the last chunk of a sequence to the first, seeded by dht (or 0); the result
// after the first chunk is dh0. The pages' backward adapters hand this reverse-order pass to
// a native `chunk_gated_delta_rule_bwd_dhu` stage (KDA coverage page, `_AscendCKDAStages`
// backward); the recurrence above is the exact adjoint of the forward chunk loop.
//
// GB300 mapping mirrors the forward chain: one CTA per (sequence, head); dS is held
// transposed in TMEM (lane v = column v of dS) in fp32, in two buffers that alternate by chunk
// step, and the dv_new product reads it there as its A operand (kind::tf32 reads the upper 19
// bits). While that product runs, the chain warps write gam dS' into the other buffer (and the
// feature-major kernel's copy of dS'), where the step's two other products accumulate. dO^T is
// staged in TMEM a step ahead; dv_new^T stays in its accumulator (double-buffered by step) and
// is the A operand of the W^T product, issued with B negated. The chunk tiles (Kt, Aqk^T,
// Qt^T, W^T, double-buffered) are TMA-loaded SW128 B operands; every product is a 128-lane
// tf32 MMA. So a step's serial path is the dv_new product and the W^T product, issued back to
// back by one thread; the chain warps' decay runs beside the first. Eight chain warps, one
// producer warp; all waits bounded.
//
// As in the forward chain, a CTA runs one segment (segments counted from the sequence's end)
// in full, or as the segment's adjoint map: from the identity with dO = 0 (M^T, the products
// of dO and their tiles left out) or from zero (the offset), with no saves.
#include "common.cuh"
#include "umma.cuh"

namespace gdn {

namespace {

constexpr int kChainThreads = 256;
constexpr int kThreads = kChainThreads + 32;
constexpr uint32_t kStage = 114688;                  // one chunk's tiles
constexpr uint32_t kOffKt = 0;                       // [t][k]  4 panels x 64 rows   (32 KB)
constexpr uint32_t kOffAqkT = 32768;                 // [t][i]  2 panels x 64 rows   (16 KB)
constexpr uint32_t kOffQtT = 49152;                  // [k][i]  2 panels x 128 rows  (32 KB)
constexpr uint32_t kOffWT = 81920;                   // [k][t]  2 panels x 128 rows  (32 KB)
constexpr uint32_t kSmemBytes = 2 * kStage + 1024;
// TMEM columns: two dS buffers (the one entering chunk step j is buffer j % 2; the decayed
// gradient and the step's updates go to the other), then dv_new and dO^T, each
// double-buffered by step parity.
__device__ __forceinline__ uint32_t tm(int j) { return uint32_t(j & 1) * 128; }
__device__ __forceinline__ uint32_t tdv(int j) { return 256 + uint32_t(j & 1) * 64; }
__device__ __forceinline__ uint32_t tdo(int j) { return 384 + uint32_t(j & 1) * 64; }

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Loads this thread's 32 dO values (token columns [t0, t0+32) of lane v) for chunk c, two
// bf16 per 32-bit register (rows past the chunk read as zero).
__device__ __forceinline__ void load_dO(const RevChainParams& p, int c, int h, int v, int t0, uint32_t* d) {
  const ChunkEntry ch = p.chunks[c];
  const unsigned short* src =
      reinterpret_cast<const unsigned short*>(p.dO) + (size_t(ch.x + t0) * p.H + h) * kD + v;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t lo = (t0 + 2 * i < ch.y) ? src[size_t(2 * i) * p.H * kD] : 0u;
    const uint32_t hi = (t0 + 2 * i + 1 < ch.y) ? src[size_t(2 * i + 1) * p.H * kD] : 0u;
    d[i] = lo | (hi << 16);
  }
}

// dS' of chunk c (the gradient w.r.t. the state leaving it; buffer tm(j), which the step's
// dv_new product reads as it is) times the chunk's decay gam, into buffer tm(j+1), where the
// step's products then accumulate; this thread: lane v, state columns [k0, k0+64). With dh_save
// the feature-major backward kernel's copy of dS' (bf16) is written from the same registers.
__device__ __forceinline__ void rev_decay_into(const RevChainParams& p, __nv_bfloat16* dh_save, int c, int h, int v, int k0,
                                               uint32_t tl, int j, float g0) {
  const size_t tile = size_t(c) * p.H + h;
  float s[64];
  tmem_ld64(tl + tm(j) + k0, s);
  tmem_wait_ld_regs(s);
  if (dh_save) store_col_bf16<64>(dh_save + tile * kD * kD + size_t(k0) * kD, s, v);
  if (p.kda) {
    const float4* gam = reinterpret_cast<const float4*>(p.gam + tile * kD + k0);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float4 g4 = gam[e];
      s[4 * e] *= g4.x;
      s[4 * e + 1] *= g4.y;
      s[4 * e + 2] *= g4.z;
      s[4 * e + 3] *= g4.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 64; ++e) s[e] *= g0;
  }
  tmem_st32(tl + tm(j + 1) + k0, s);
  tmem_st32(tl + tm(j + 1) + k0 + 32, s + 32);
}

// dO^T of the chunk handled at step j (prefetched into `d`: this thread's token columns
// [t0, t0+32), two bf16 per register) into its TMEM slot tdo(j), a step ahead of its products.
__device__ __forceinline__ void stage_do(uint32_t tl, int j, int t0, const uint32_t* d) {
  float df[32];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    df[2 * i] = __uint_as_float(d[i] << 16);
    df[2 * i + 1] = __uint_as_float(d[i] & 0xffff0000u);
  }
  tmem_st32(tl + tdo(j) + t0, df);
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    k_chain_bwd(const __grid_constant__ CUtensorMap mKt, const __grid_constant__ CUtensorMap mAqkT,
                const __grid_constant__ CUtensorMap mQtT, const __grid_constant__ CUtensorMap mWT,
                const __grid_constant__ CUtensorMap mdO, const RevChainParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1k(smem_raw);
  __shared__ uint64_t full[2], mma1, mma2, doready, mready;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y + p.hg0, H = p.H;
  // which segment of which sequence (processing order: from the end), and how
  const SegPlan& sp = p.sp;
  const int runs = runs_per_seq(sp.maxS, sp.pass);
  const int n = blockIdx.x / runs, slot = blockIdx.x % runs;
  const SeqEntry seq = p.seqs[n];
  const int ns = (seq.y + sp.L - 1) / sp.L;
  int seg = 0, mode = kRunFull;
  if (!decode_run(slot, sp.pass, ns, &seg, &mode)) return;
  const int lo = (ns - 1 - seg) * sp.L;          // first chunk of the segment within the sequence
  const int nc = min(sp.L, seq.y - lo);
  const int last = seq.x + lo + nc - 1;
  const bool outs = mode == kRunFull;            // saves and dh0
  const bool use_do = mode != kRunMapM;          // dO enters the recurrence
  const size_t slot_base = size_t(n) * sp.maxS;

  if (warp == 0) tmem_alloc(&tslot, 512);
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(&mma1, 1);
    mbar_init(&mma2, 1);
    mbar_init(&doready, kChainThreads);
    mbar_init(&mready, kChainThreads);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;

  if (warp == kChainThreads / 32) {
    if (lane == 0) {
      auto load = [&](int c, int st) {
        uint8_t* base = sm + st * kStage;
        const int y64 = (c * H + h) * kC, y128 = (c * H + h) * kD;
        mbar_expect_tx(&full[st], use_do ? kStage : 65536u);
        for (int pp = 0; pp < 4; ++pp) tma_load_2d(base + kOffKt + pp * 8192, &mKt, pp * 32, y64, &full[st]);
        for (int pp = 0; pp < 2; ++pp) {
          if (use_do) {
            tma_load_2d(base + kOffAqkT + pp * 8192, &mAqkT, pp * 32, y64, &full[st]);
            tma_load_2d(base + kOffQtT + pp * 16384, &mQtT, pp * 32, y128, &full[st]);
          }
          tma_load_2d(base + kOffWT + pp * 16384, &mWT, pp * 32, y128, &full[st]);
        }
      };
      // dO rows of a chunk into L2 ahead of the chain warps' loads of them (a sequence's chunks
      // are consecutive 64-token runs, so the row follows from the last chunk's, read once)
      const int row_last = p.chunks[last].x;
      auto prefetch_do = [&](int c) {
        const int row = row_last - kC * (last - c);
        prefetch_l2_tile(&mdO, h * kD, row);
        prefetch_l2_tile(&mdO, h * kD + 64, row);
      };
      load(last, 0);
      if (nc > 1) load(last - 1, 1);
      if (use_do && nc > 1) prefetch_do(last - 1);
      if (use_do && nc > 2) prefetch_do(last - 2);
      const uint32_t id64 = idesc_tf32(128, 64), id128 = idesc_tf32(128, 128);
      for (int j = 0; j < nc; ++j) {
        const int c = last - j, st = j & 1;
        const uint32_t par = j & 1;
        const uint32_t base = smem_u32(sm + st * kStage);
        if (!mbar_wait(&full[st], (j >> 1) & 1, &abort_flag, p.status, kDevTimeoutTma)) break;
        // dO^T of this chunk is in its TMEM slot (staged a step ahead); at the first step this
        // also means the seed gradient is in its buffer
        if ((use_do || j == 0) && !mbar_wait(&doready, par, &abort_flag, p.status, kDevTimeoutSync)) break;
        tc_fence_after();
        // dv_new^T = dO^T Aqk + dS'^T Kt^T, with dS' read from its buffer as it is
        if (use_do)
          for (int s = 0; s < 8; ++s) mma_tf32_ts(tb + tdv(j), tb + tdo(j) + s * 8, desc_kmajor(base + kOffAqkT, 8192, s), id64, s > 0);
        for (int s = 0; s < 16; ++s)
          mma_tf32_ts(tb + tdv(j), tb + tm(j) + s * 8, desc_kmajor(base + kOffKt, 8192, s), id64, use_do || s > 0);
        mma_commit(&mma1);
        // dS^T += dO^T Qt, once the other buffer holds gam dS'^T
        if (!mbar_wait(&mready, par, &abort_flag, p.status, kDevTimeoutSync)) break;
        tc_fence_after();
        if (use_do)
          for (int s = 0; s < 8; ++s) mma_tf32_ts(tb + tm(j + 1), tb + tdo(j) + s * 8, desc_kmajor(base + kOffQtT, 16384, s), id128, true);
        if (!mbar_wait(&mma1, par, &abort_flag, p.status, kDevTimeoutMma)) break;
        tc_fence_after();
        // dS^T -= dv_new^T W, dv_new read from its accumulator (B negated)
        for (int s = 0; s < 8; ++s)
          mma_tf32_ts(tb + tm(j + 1), tb + tdv(j) + s * 8, desc_kmajor(base + kOffWT, 16384, s), id128 | (1u << 14), true);
        mma_commit(&mma2);
        if (use_do && j + 3 < nc) prefetch_do(c - 3);
        if (!mbar_wait(&mma2, par, &abort_flag, p.status, kDevTimeoutMma)) break;
        if (j + 2 < nc) load(c - 2, st);
      }
    }
  } else if (warp < kChainThreads / 32) {
    const int v = tid & 127, half = tid >> 7;
    const uint32_t tl = tb + tmem_lane_base(warp);
    const int k0 = 64 * half, t0 = 32 * half;
    __nv_bfloat16* dh_save = outs ? p.dh_save : nullptr;
    float* dvn_save = outs ? p.dvn_save : nullptr;
    {
      // seed: dht, a composed segment seed, the identity (map M) or zero
      const float* src = nullptr;
      if (mode == kRunFull)
        src = seg == 0 ? (p.dht ? p.dht + (size_t(n) * H + h) * kD * kD : nullptr)
                       : sp.E + ((slot_base + seg) * H + h) * kD * kD;
      float buf[64];
      if (src) src += size_t(k0) * kD + v;
#pragma unroll
      for (int e = 0; e < 64; ++e)
        buf[e] = src ? src[size_t(e) * kD] : (mode == kRunMapM && k0 + e == v ? 1.f : 0.f);
      tmem_st32(tl + tm(0) + k0, buf);
      tmem_st32(tl + tm(0) + k0 + 32, buf + 32);
      tmem_wait_st();
    }
    bool alive = true;
    // dO of the chunk after the one being staged is loaded a whole step ahead of its staging
    uint32_t dnext[16];
    if (use_do) {
      load_dO(p, last, h, v, t0, dnext);
      stage_do(tl, 0, t0, dnext);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&doready);   // the seed (and the first chunk's dO^T) are in TMEM
    if (use_do && nc > 1) load_dO(p, last - 1, h, v, t0, dnext);
    float g_cur = p.kda ? 0.f : p.gam[(size_t(last) * H + h) * kD];
    for (int j = 0; j < nc; ++j) {
      const int c = last - j;
      const uint32_t par = j & 1;
      const size_t tile = size_t(c) * H + h;
      // next chunk's scalar gate, loaded a step ahead of its use
      const float g_next = (j + 1 < nc && !p.kda) ? p.gam[(size_t(c - 1) * H + h) * kD] : 0.f;
      // the decayed gradient into the other buffer while the dv_new product reads dS'
      rev_decay_into(p, dh_save, c, h, v, k0, tl, j, g_cur);
      g_cur = g_next;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&mready);
      if (!mbar_wait(&mma1, par, &abort_flag, p.status, kDevTimeoutMma)) { alive = false; break; }
      tc_fence_after();
      if (dvn_save) {
        // dv_new for the feature-major kernel (rounded to tf32); its buffer is rewritten two
        // steps on, after this thread's next mready arrival
        float r[32];
        tmem_ld32(tl + tdv(j) + t0, r);
        tmem_wait_ld_regs(r);
        float* dv = dvn_save + tile * kTileW + size_t(t0) * kD + v;
#pragma unroll
        for (int t = 0; t < 32; ++t) dv[size_t(t) * kD] = to_tf32(r[t]);
      }
      // the next chunk's dO^T into the other slot (its last readers, the previous step's
      // products, completed before that step's final wait)
      if (use_do && j + 1 < nc) {
        stage_do(tl, j + 1, t0, dnext);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&doready);
        if (j + 2 < nc) load_dO(p, c - 2, h, v, t0, dnext);
      }
      if (!mbar_wait(&mma2, par, &abort_flag, p.status, kDevTimeoutMma)) { alive = false; break; }
      tc_fence_after();
    }
    // exit gradient: dh0, the next segment's seed (pass 0), or the segment's map
    float* dst = nullptr;
    if (mode == kRunFull) {
      if (seg == ns - 1) dst = p.dh0 ? p.dh0 + (size_t(n) * H + h) * kD * kD : nullptr;
      else if (sp.pass == 0) dst = sp.E + ((slot_base + seg + 1) * H + h) * kD * kD;
    } else if (mode == kRunMapM) {
      dst = sp.Phi + ((slot_base + seg) * H + h) * kD * kD;
    } else {
      dst = sp.Bm + ((slot_base + seg) * H + h) * kD * kD;
    }
    if (alive && dst) {  // the loop's last mma2 wait covers the final update
      float s[64];
      tmem_ld64(tl + tm(nc) + k0, s);
      tmem_wait_ld_regs(s);
      const size_t off = size_t(k0) * kD + v;
      if (mode == kRunMapM) {
        // the map transposed: this thread's row v of M^T, columns k0 .. k0+63 (the compose
        // step reads four rows of M at a time as one 16-byte load)
        float4* row = reinterpret_cast<float4*>(dst + size_t(v) * kD + k0);
#pragma unroll
        for (int e = 0; e < 16; ++e) row[e] = make_float4(s[4 * e], s[4 * e + 1], s[4 * e + 2], s[4 * e + 3]);
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) dst[off + size_t(e) * kD] = s[e];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 512);
}

cudaError_t launch_chain_bwd(const CUtensorMap& mKt, const CUtensorMap& mAqkT, const CUtensorMap& mQtT,
                             const CUtensorMap& mWT, const CUtensorMap& mdO, const RevChainParams& p,
                             cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_chain_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(p.N * runs_per_seq(p.sp.maxS, p.sp.pass), p.hgn);
  k_chain_bwd<<<grid, kThreads, kSmemBytes, s>>>(mKt, mAqkT, mQtT, mWT, mdO, p);
  return cudaGetLastError();
}

}  // namespace gdn
