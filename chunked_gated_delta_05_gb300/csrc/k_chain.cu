// Chain kernel: the serial inter-chunk state recurrence fused with the chunk output.
//
// Per chunk, with S the K x V state entering it (the chunk loop of the eager reference
// `torch_chunk_gated_delta_rule`, hyper-parallel GDN Diff Coverage page):
//   v_new = U - W S
//   o     = Qt S + Aqk v_new
//   S     = diag(gam) S + k~^T v_new,     k~ = keys decayed to the chunk end (KtT = k~^T)
// (gam is exp(G_last): a scalar for GDN, one value per key row for KDA.)
//
// GB300 mapping: one CTA per (sequence, head). The state lives in TMEM, transposed: S^T
// (V x K), lane v = column v of S, as one fp32 copy that the MMAs read as their TMEM-resident
// A operand (kind::tf32, which reads the operand's upper 19 bits; a CPU emulation of the chunked
// algorithm gives the same state and output errors as with a round-to-nearest copy). Two state
// buffers alternate by chunk parity. The chunk tiles from the prepare kernel are TMA-loaded
// SW128 B operands:
//   [P | O] = S^T [W; Qt]^T  (one N=128 product: P = S^T W^T, O = S^T Qt^T)  -- on the chain
//   S'^T    = S^T diag(gam)  (the chain warps, into the other buffer, while the product reads S)
//   v_new^T = U^T - P        (written over P in TMEM)
//   S'^T   += v_new^T KtT^T                                -- on the serial chain
//   O      += v_new^T Aqk^T                                -- off the chain, issued after
// The decay (and the backward's bf16 copy of the entry state, taken from the same registers)
// overlaps the product. The issuing thread starts the next chunk's product as soon as the
// state update completes. P/v_new and O are double-buffered in TMEM by chunk parity; a chunk's
// output is read out while the next chunk's state update runs, and the product two chunks on
// waits for that read. Eight chain warps share the TMEM lanes (two threads per lane, each on
// half of the columns); warp 8 streams the tiles with TMA (KtT/Aqk double-buffered) and issues
// the MMAs from one thread. All waits bounded.
//
// A CTA runs one segment of a sequence's chunks in one of three modes (the segmented chain
// of common.cuh): in full (from the true entry state, with the output and the backward
// saves), or as the segment's affine map, from the identity with U = 0 (M) or from zero
// (B), with no outputs and the output products, Qt and Aqk left out. In M mode v_new = -P,
// so the state update reads P from its accumulator with B negated (as the reverse chain
// reads dv_new), and the chain warps' v_new pass leaves the serial path.
#include "common.cuh"
#include "umma.cuh"

namespace gdn {

namespace {

constexpr int kChainThreads = 256;            // 8 warps: lane v = tid % 128, half = tid / 128
constexpr int kThreads = kChainThreads + 32;  // + producer warp
// shared memory tile offsets (bytes, 1024-aligned)
constexpr uint32_t kOffWQ = 0;         // 4 panels x 128 rows x 128 B: rows 0-63 W [t][k], 64-127 Qt [t][k]
constexpr uint32_t kOffU = 65536;      // 4 panels x [64][32] fp32, no swizzle
constexpr uint32_t kOffG3 = 98304;     // 2 stages x {KtT 32 KB (2 panels x 128 rows), Aqk 16 KB}
constexpr uint32_t kG3Stage = 49152;
constexpr uint32_t kSmemBytes = kOffG3 + 2 * kG3Stage + 1024;
// TMEM columns: two state buffers, then per chunk parity [P, later v_new | O]. The state
// entering chunk j lives in buffer j % 2; the decayed state and the update go to the other.
constexpr uint32_t kTB = 256;
__device__ __forceinline__ uint32_t ts(int j) { return uint32_t(j & 1) * 128; }
__device__ __forceinline__ uint32_t tpv(int j) { return kTB + uint32_t(j & 1) * 128; }
__device__ __forceinline__ uint32_t tout(int j) { return kTB + uint32_t(j & 1) * 128 + 64; }

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// The state entering chunk j (buffer ts(j); this thread: lane v, state columns [k0, k0+64))
// times chunk c's end decay gam, into buffer ts(j+1), where the chunk's state update then adds
// k~^T v_new. It runs while the chunk's product reads buffer ts(j). With h_save the entry
// state also goes to the backward's save (bf16) from the same registers.
__device__ __forceinline__ void chain_decay_into(const ChainParams& p, int c, int h, int v, int k0, uint32_t tl,
                                                 int j, float g0, __nv_bfloat16* h_save) {
  float s[64];
  tmem_ld64(tl + ts(j) + k0, s);
  tmem_wait_ld_regs(s);
  if (h_save) store_col_bf16<64>(h_save + (size_t(c) * p.H + h) * kD * kD + size_t(k0) * kD, s, v);
  if (p.kda) {
    const float4* gam = reinterpret_cast<const float4*>(p.gam + (size_t(c) * p.H + h) * kD + k0);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float4 g4 = gam[e];
      float* x = s + 4 * e;
      x[0] *= g4.x;
      x[1] *= g4.y;
      x[2] *= g4.z;
      x[3] *= g4.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 64; ++e) s[e] *= g0;
  }
  tmem_st32(tl + ts(j + 1) + k0, s);
  tmem_st32(tl + ts(j + 1) + k0 + 32, s + 32);
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    k_chain_fwd(const __grid_constant__ CUtensorMap mW, const __grid_constant__ CUtensorMap mQt,
                const __grid_constant__ CUtensorMap mKtT, const __grid_constant__ CUtensorMap mAqk,
                const __grid_constant__ CUtensorMap mU, const ChainParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1k(smem_raw);
  __shared__ uint64_t full1, full1b, full2, full3[2], mma1, mma2, mma3, sready, vready, oread;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y + p.hg0, H = p.H;
  // which segment of which sequence, and how
  const SegPlan& sp = p.sp;
  const int runs = runs_per_seq(sp.maxS, sp.pass);
  const int n = blockIdx.x / runs, slot = blockIdx.x % runs;
  const SeqEntry seq = p.seqs[n];
  const int ns = (seq.y + sp.L - 1) / sp.L;
  int seg = 0, mode = kRunFull;
  if (!decode_run(slot, sp.pass, ns, &seg, &mode)) return;
  const int first = seq.x + seg * sp.L, nc = min(sp.L, seq.y - seg * sp.L);
  const bool outs = mode == kRunFull;     // output, saves and the output products
  const bool use_u = mode != kRunMapM;    // U enters v_new
  const size_t slot_base = size_t(n) * sp.maxS;

  if (warp == 0) tmem_alloc(&tslot, 512);
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&full1, 1);
    mbar_init(&full1b, 1);
    mbar_init(&full2, 1);
    mbar_init(&full3[0], 1);
    mbar_init(&full3[1], 1);
    mbar_init(&mma1, 1);
    mbar_init(&mma2, 1);
    mbar_init(&mma3, 1);
    mbar_init(&sready, kChainThreads);
    mbar_init(&vready, kChainThreads);
    mbar_init(&oread, kChainThreads);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;

  if (warp == kChainThreads / 32) {
    if (lane == 0) {
      // ---------------- producer + MMA issuer ----------------
      const uint32_t sWQ = smem_u32(sm + kOffWQ);
      auto load_g1 = [&](int c) {
        const int y = (c * H + h) * kC;
        mbar_expect_tx(&full1, outs ? 65536u : 32768u);
        for (int pp = 0; pp < 4; ++pp) {
          tma_load_2d(sm + kOffWQ + pp * 16384, &mW, pp * 32, y, &full1);
          if (outs) tma_load_2d(sm + kOffWQ + pp * 16384 + 8192, &mQt, pp * 32, y, &full1);
        }
      };
      auto load_g2 = [&](int c) {
        const int y = (c * H + h) * kC;
        mbar_expect_tx(&full2, 32768u);
        for (int pp = 0; pp < 4; ++pp) tma_load_2d(sm + kOffU + pp * 8192, &mU, pp * 32, y, &full2);
      };
      auto load_g3 = [&](int c, int st) {
        uint8_t* base = sm + kOffG3 + st * kG3Stage;
        mbar_expect_tx(&full3[st], outs ? 49152u : 32768u);
        for (int pp = 0; pp < 2; ++pp) {
          tma_load_2d(base + pp * 16384, &mKtT, pp * 32, (c * H + h) * kD, &full3[st]);
          if (outs) tma_load_2d(base + 32768 + pp * 8192, &mAqk, pp * 32, (c * H + h) * kC, &full3[st]);
        }
      };
      // M mode: W double-buffered in the rows Qt takes in full mode (full1 for even steps,
      // full1b for odd ones), so each W copy has two steps to land
      auto load_w = [&](int c, int b) {
        uint64_t* bar = b ? &full1b : &full1;
        mbar_expect_tx(bar, 32768u);
        for (int pp = 0; pp < 4; ++pp) tma_load_2d(sm + kOffWQ + pp * 16384 + b * 8192, &mW, pp * 32, (c * H + h) * kC, bar);
      };
      if (mode == kRunMapM) {
        load_w(first, 0);
        if (nc > 1) load_w(first + 1, 1);
      } else {
        load_g1(first);
      }
      if (use_u) load_g2(first);
      load_g3(first, 0);
      if (nc > 1) load_g3(first + 1, 1);
      const uint32_t id64 = idesc_tf32(128, 64), id128 = idesc_tf32(128, 128);
      const uint32_t id_first = outs ? id128 : id64;  // [P | O] or P alone
      const uint32_t id128_negb = id128 | (1u << 14);   // B negated
      // the chain warps have written the entry state
      bool alive = mbar_wait(&sready, 0, &abort_flag, p.status, kDevTimeoutSync);
      for (int j = 0; j < nc && alive; ++j) {
        const uint32_t par = j & 1;
        const int c = first + j, st = j & 1;
        const uint32_t tPV = tb + tpv(j), tO = tb + tout(j);
        const uint32_t sKtT = smem_u32(sm + kOffG3 + st * kG3Stage), sAqk = sKtT + 32768;
        if (mode == kRunMapM) {
          if (!mbar_wait(par ? &full1b : &full1, (j >> 1) & 1, &abort_flag, p.status, kDevTimeoutTma)) break;
          // U = 0, so v_new = -P: the update reads the product's accumulator itself, with B
          // negated, issued right behind it (the MMAs run in issue order), as the reverse chain
          // does; the chain warps only decay the state
          tc_fence_after();
          for (int s = 0; s < 16; ++s)
            mma_tf32_ts(tPV, tb + ts(j) + s * 8, desc_kmajor(sWQ + par * 8192, 16384, s), id64, s > 0);
          mma_commit(&mma1);
          if (j > 0) {
            if (!mbar_wait(&mma3, par ^ 1u, &abort_flag, p.status, kDevTimeoutMma)) break;
            if (j + 1 < nc) load_g3(c + 1, st ^ 1);
          }
          if (!mbar_wait(&full3[st], (j >> 1) & 1, &abort_flag, p.status, kDevTimeoutTma)) break;
          if (!mbar_wait(&vready, par, &abort_flag, p.status, kDevTimeoutSync)) break;
          tc_fence_after();
          for (int s = 0; s < 8; ++s) mma_tf32_ts(tb + ts(j + 1), tPV + s * 8, desc_kmajor(sKtT, 16384, s), id128_negb, true);
          mma_commit(&mma2);
          mma_commit(&mma3);
          // the product has read this buffer's W: the tile two chunks on may replace it
          if (!mbar_wait(&mma1, par, &abort_flag, p.status, kDevTimeoutMma)) break;
          if (j + 2 < nc) load_w(c + 2, par);
          if (!mbar_wait(&mma2, par, &abort_flag, p.status, kDevTimeoutMma)) break;
          continue;
        }
        if (!mbar_wait(&full1, par, &abort_flag, p.status, kDevTimeoutTma)) break;
        // the product overwrites the output of chunk j - 2: the chain warps have read it
        if (outs && p.o && j >= 2 && !mbar_wait(&oread, par, &abort_flag, p.status, kDevTimeoutSync)) break;
        tc_fence_after();
        for (int s = 0; s < 16; ++s) mma_tf32_ts(tPV, tb + ts(j) + s * 8, desc_kmajor(sWQ, 16384, s), id_first, s > 0);
        mma_commit(&mma1);
        // the previous chunk's output product has read its KtT / Aqk stage: refill it two chunks on
        if (j > 0) {
          if (!mbar_wait(&mma3, par ^ 1u, &abort_flag, p.status, kDevTimeoutMma)) break;
          if (j + 1 < nc) load_g3(c + 1, st ^ 1);
        }
        if (!mbar_wait(&mma1, par, &abort_flag, p.status, kDevTimeoutMma)) break;
        if (j + 1 < nc) load_g1(c + 1);
        if (!mbar_wait(&full3[st], (j >> 1) & 1, &abort_flag, p.status, kDevTimeoutTma)) break;
        // the chain warps have decayed the state into the other buffer and written v_new
        if (!mbar_wait(&vready, par, &abort_flag, p.status, kDevTimeoutSync)) break;
        tc_fence_after();
        for (int s = 0; s < 8; ++s) mma_tf32_ts(tb + ts(j + 1), tPV + s * 8, desc_kmajor(sKtT, 16384, s), id128, true);
        mma_commit(&mma2);
        if (outs)
          for (int s = 0; s < 8; ++s) mma_tf32_ts(tO, tPV + s * 8, desc_kmajor(sAqk, 8192, s), id64, true);
        mma_commit(&mma3);
        if (j + 1 < nc && use_u) load_g2(c + 1);  // the chain warps read U into registers before v_new
        // the next chunk's product goes out as soon as the state update is complete
        if (!mbar_wait(&mma2, par, &abort_flag, p.status, kDevTimeoutMma)) break;
      }
    }
  } else if (warp < kChainThreads / 32) {
    // ---------------- chain warps: lane v of S^T, column half `half` ----------------
    const int v = tid & 127, half = tid >> 7;
    const uint32_t lb = tmem_lane_base(warp);
    const float* sU = reinterpret_cast<const float*>(sm + kOffU);
    const int k0 = 64 * half;  // state columns handled by this thread
    const int t0 = 32 * half;  // token columns handled by this thread
    __nv_bfloat16* h_save = outs ? p.h_save : nullptr;
    float* vnew_save = outs ? p.vnew_save : nullptr;
    __nv_bfloat16* o = outs ? p.o : nullptr;
    {
      // entry state: the initial state, a composed segment entry, the identity (map M) or zero
      const float* src = nullptr;
      if (mode == kRunFull)
        src = seg == 0 ? (p.h0 ? p.h0 + (size_t(n) * H + h) * kD * kD : nullptr) : sp.E + ((slot_base + seg) * H + h) * kD * kD;
      float buf[64];
      if (src) src += size_t(k0) * kD + v;
#pragma unroll
      for (int e = 0; e < 64; ++e)
        buf[e] = src ? src[size_t(e) * kD] : (mode == kRunMapM && k0 + e == v ? 1.f : 0.f);
      tmem_st32(tb + lb + ts(0) + k0, buf);
      tmem_st32(tb + lb + ts(0) + k0 + 32, buf + 32);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&sready);
      if (h_save) {
        // the entry state of the first chunk, from the registers (identical to what was stored)
        store_col_bf16<64>(h_save + (size_t(first) * H + h) * kD * kD + size_t(k0) * kD, buf, v);
      }
    }
    bool alive = true;
    float g_cur = p.kda ? 0.f : p.gam[(size_t(first) * H + h) * kD];
    // the output of chunk jj: lane pairs (v, v^1) swap halves so each lane stores two adjacent
    // bf16 of a row (the even lane rows t0..t0+15, the odd lane rows t0+16..t0+31); the chain
    // warps arrive on oread once the tile is in registers (the product two chunks on rewrites it)
    auto out_epilogue = [&](int jj, bool signal) {
      const ChunkEntry ch = p.chunks[first + jj];
      float r[32];
      tmem_ld32(tb + lb + tout(jj) + t0, r);
      tmem_wait_ld_regs(r);
      if (signal) {
        tc_fence_before();
        mbar_arrive(&oread);
      }
      const int odd = v & 1;
      __nv_bfloat162* op = reinterpret_cast<__nv_bfloat162*>(o + (size_t(ch.x + t0 + 16 * odd) * H + h) * kD + (v & ~1));
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float mine = odd ? r[16 + t] : r[t];
        const float give = odd ? r[t] : r[16 + t];
        const float other = __shfl_xor_sync(0xffffffffu, give, 1);
        const __nv_bfloat162 pr = odd ? __floats2bfloat162_rn(other, mine) : __floats2bfloat162_rn(mine, other);
        if (t0 + 16 * odd + t < ch.y) op[size_t(t) * H * kD / 2] = pr;
      }
    };
    for (int j = 0; j < nc; ++j) {
      const uint32_t par = j & 1;
      const int c = first + j;
      const size_t tile = size_t(c) * H + h;
      // next chunk's scalar gate, loaded a chunk ahead of its use
      const float g_next = (j + 1 < nc && !p.kda) ? p.gam[(size_t(c + 1) * H + h) * kD] : 0.f;
      // the decayed state into the other buffer while this chunk's product reads the state (the
      // segment's first entry state was saved from the registers that wrote it)
      chain_decay_into(p, c, h, v, k0, tb + lb, j, g_cur, j > 0 ? h_save : nullptr);
      if (mode == kRunMapM) {
        // the update negates P itself: signal the decayed state only
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&vready);
        g_cur = g_next;
        if (!mbar_wait(&mma2, par, &abort_flag, p.status, kDevTimeoutMma)) { alive = false; break; }
        tc_fence_after();
        continue;
      }
      if (use_u && !mbar_wait(&full2, par, &abort_flag, p.status, kDevTimeoutTma)) { alive = false; break; }
      if (!mbar_wait(&mma1, par, &abort_flag, p.status, kDevTimeoutMma)) { alive = false; break; }
      // the previous chunk's intra-chunk output product was issued before this product
      if (o && j > 0 && !mbar_wait(&mma3, par ^ 1u, &abort_flag, p.status, kDevTimeoutMma)) { alive = false; break; }
      tc_fence_after();
      {
        float r[32];
        tmem_ld32(tb + lb + tpv(j) + t0, r);
        float u[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) u[t] = use_u ? sU[(v >> 5) * 2048 + (t0 + t) * 32 + (v & 31)] : 0.f;
        tmem_wait_ld_regs(r);
#pragma unroll
        for (int t = 0; t < 32; ++t) r[t] = to_tf32(u[t] - r[t]);
        tmem_st32(tb + lb + tpv(j) + t0, r);
        tmem_wait_st();   // the decayed state's stores as well
        tc_fence_before();
        mbar_arrive(&vready);
        if (vnew_save) {
          float* vsave = vnew_save + tile * kTileW + size_t(t0) * kD + v;
#pragma unroll
          for (int t = 0; t < 32; ++t) vsave[size_t(t) * kD] = r[t];
        }
      }
      // the previous chunk's output, while this chunk's state update runs
      if (o && j > 0) out_epilogue(j - 1, true);
      g_cur = g_next;
      if (!mbar_wait(&mma2, par, &abort_flag, p.status, kDevTimeoutMma)) { alive = false; break; }
      tc_fence_after();
    }
    if (o && alive) {
      if (mbar_wait(&mma3, (nc - 1) & 1, &abort_flag, p.status, kDevTimeoutMma)) {
        tc_fence_after();
        out_epilogue(nc - 1, false);
      } else {
        alive = false;
      }
    }
    // exit state: the final state, the next segment's entry (pass 0), or the segment's map
    float* dst = nullptr;
    if (mode == kRunFull) {
      if (seg == ns - 1) dst = p.hT ? p.hT + (size_t(n) * H + h) * kD * kD : nullptr;
      else if (sp.pass == 0) dst = sp.E + ((slot_base + seg + 1) * H + h) * kD * kD;
    } else if (mode == kRunMapM) {
      dst = sp.Phi + ((slot_base + seg) * H + h) * kD * kD;
    } else {
      dst = sp.Bm + ((slot_base + seg) * H + h) * kD * kD;
    }
    if (alive && dst) {  // the loop's last mma2 wait covers the final state update
      float s[64];
      tmem_ld64(tb + lb + ts(nc) + k0, s);
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

cudaError_t launch_chain_fwd(const CUtensorMap& mW, const CUtensorMap& mQt, const CUtensorMap& mKtT,
                             const CUtensorMap& mAqk, const CUtensorMap& mU, const ChainParams& p,
                             cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_chain_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(p.N * runs_per_seq(p.sp.maxS, p.sp.pass), p.hgn);
  k_chain_fwd<<<grid, kThreads, kSmemBytes, s>>>(mW, mQt, mKtT, mAqk, mU, p);
  return cudaGetLastError();
}

}  // namespace gdn
