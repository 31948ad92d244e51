// Blackwell (sm_103a) building blocks: tcgen05 tensor-core MMA with TMEM accumulators,
// TMA tile copies, mbarriers with bounded waits, and the shared-memory operand layout.
//
// Operand layout convention used by every kernel of this library ("SW128 K-major"):
// an operand tile of R rows x Kc columns is stored as Kc*es/128 panels, each panel R rows of
// 128 bytes, 8-row groups 1024 bytes apart, the 16-byte chunks of row r XOR-permuted by
// (r % 8) (the 128-byte swizzle that TMA's CU_TENSOR_MAP_SWIZZLE_128B produces). Panels
// start on 1024-byte boundaries. Rows are the M (or N) index of the MMA, columns its K index.
// An "MN-major" tile (only for TMA-loaded bf16 tiles used as the B operand) is the same
// bytes read the other way: rows are the K index, each 128-byte row holds 64 N entries.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda.h>
#include <cuda_bf16.h>

namespace gdn {

// ------------------------------------------------------------------ error flag codes
// Device kernels never trap; a bounded wait that runs out records one of these in the
// caller-visible status word and the kernel winds down.
enum DevErr : int {
  kDevOk = 0,
  kDevTimeoutTma = 1,
  kDevTimeoutMma = 2,
  kDevTimeoutSync = 3,
  kDevGateRange = 5,  // a per-channel gate dropped faster than the kernels support (GDN_ERANGE)
};

// Spin limit for every mbarrier wait, in nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` to complete. Gives up after kWaitLimitNs, records `code` in
// *abort (shared) and *status (global), and returns false. Once *abort is set every later
// wait returns false at once, so all threads reach the kernel's exit path.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* status, int code,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (*abort) return false;
    if (mbar_try(bar, parity)) return true;
    if (globaltimer() - t0 > limit_ns) {
      *abort = 1;
      if (status) atomicCAS(status, 0, code);
      return false;
    }
  }
}
// Bounded wait that ignores the abort flag: an aborting CTA uses it to let its own copies and
// MMAs that are already in flight finish before it frees their destinations. False after
// `limit_ns` without completion.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity,
                                           unsigned long long limit_ns = kWaitLimitNs) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try(bar, parity))
    if (globaltimer() - t0 > limit_ns) return false;
  return true;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, int x, int y, const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
               ::"l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// The committed stores have finished reading their shared-memory sources (which may be reused).
__device__ __forceinline__ void tma_store_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Untiled bulk copy global -> shared of `bytes` (a multiple of 16; both addresses 16-byte
// aligned), completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Fetch `bytes` (a multiple of 16, 16-byte aligned source) into L2 ahead of use; no
// completion to wait for.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

// L2 prefetch of one box of a tensor map (no shared memory involved).
__device__ __forceinline__ void prefetch_l2_tile(const CUtensorMap* m, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
               ::"l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y)
               : "memory");
}

// The CTA that starts about one wave after this one when every SM runs one CTA at a time
// (linear block index + `sms`), as (x, y) of a 2-D grid; false past the end of the grid.
__device__ __forceinline__ bool next_wave_block(int sms, int* x, int* y) {
  const long long next = (long long)blockIdx.y * gridDim.x + blockIdx.x + sms;
  if (next >= (long long)gridDim.x * gridDim.y) return false;
  *x = int(next % gridDim.x);
  *y = int(next / gridDim.x);
  return true;
}

// Generic-proxy shared-memory writes -> visible to the async proxy (tensor core, TMA).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Lane base for the calling warp: a warp may only touch TMEM lanes 32*(warp%4) .. +31.
__device__ __forceinline__ uint32_t tmem_lane_base(int warp) { return uint32_t((warp & 3) * 32) << 16; }

// 32 lanes x 16 consecutive 32-bit columns per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* r) {
  uint32_t* u = reinterpret_cast<uint32_t*>(r);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
        "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* r) {
  const uint32_t* u = reinterpret_cast<const uint32_t*>(r);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7]),
        "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]), "r"(u[13]), "r"(u[14]), "r"(u[15])
      : "memory");
}

// 16 lanes x 64 bits, 16 repetitions (32 columns) over the warp: lane t receives row
// (t >> 2) + 8 (t & 1) of the warp's 16 lanes at columns ((t >> 1) & 1) + 2 r, r = 0..15.
__device__ __forceinline__ void tmem_ld16x64b_x16(uint32_t taddr, float* r) {
  uint32_t* u = reinterpret_cast<uint32_t*>(r);
  asm volatile(
      "tcgen05.ld.sync.aligned.16x64b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
        "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
      : "r"(taddr));
}

// 32 lanes x 32 consecutive 32-bit columns per thread (no wait; pair with tmem_wait_ld).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* r) {
  uint32_t* u = reinterpret_cast<uint32_t*>(r);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
        "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]),
        "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]),
        "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* r) {
  const uint32_t* u = reinterpret_cast<const uint32_t*>(r);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7]),
        "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]), "r"(u[13]), "r"(u[14]), "r"(u[15]),
        "r"(u[16]), "r"(u[17]), "r"(u[18]), "r"(u[19]), "r"(u[20]), "r"(u[21]), "r"(u[22]), "r"(u[23]),
        "r"(u[24]), "r"(u[25]), "r"(u[26]), "r"(u[27]), "r"(u[28]), "r"(u[29]), "r"(u[30]), "r"(u[31])
      : "memory");
}
// Wait for this thread's outstanding TMEM loads, then pin the loaded registers after the
// wait (an empty volatile asm per register) so no consumer can be scheduled above it.
template <int N>
__device__ __forceinline__ void tmem_wait_ld_regs(float (&r)[N]) {
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+f"(r[i]));
}

// 64 columns: two x32 loads issued back to back (one wait covers both).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* r) {
  tmem_ld32(taddr, r);
  tmem_ld32(taddr + 32, r + 32);
}

// ------------------------------------------------------------------ MMA descriptors
// Instruction descriptor (kind::f16 with bf16 inputs, or kind::tf32), fp32 accumulate.
// a_mn / b_mn select MN-major ("transposed") operands.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn = false, bool b_mn = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, bool a_mn = false, bool b_mn = false) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t((lbo_bytes & 0x3FFFFu) >> 4) << 16;
  d |= uint64_t((sbo_bytes & 0x3FFFFu) >> 4) << 32;
  d |= 1ull << 46;  // descriptor version for tcgen05
  d |= 2ull << 61;  // SWIZZLE_128B
  return d;
}

// Descriptor of k-step `s` (32 bytes of K per step) of a K-major SW128 tile whose panels
// are `panel_bytes` apart.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, uint32_t panel_bytes, int s) {
  return sdesc_sw128(base + uint32_t(s >> 2) * panel_bytes + uint32_t(s & 3) * 32u, 16u, 1024u);
}
// Descriptor of k-step `s` (16 K rows per step, bf16) of an MN-major SW128 tile: 128-byte
// rows indexed by K, 64 N entries per row, N-panels `panel_bytes` apart.
__device__ __forceinline__ uint64_t desc_mnmajor_bf16(uint32_t base, uint32_t panel_bytes, int s) {
  return sdesc_sw128(base + uint32_t(s) * 16u * 128u, panel_bytes, 1024u);
}

__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(uint32_t(acc))
      : "memory");
}
__device__ __forceinline__ void mma_tf32_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(uint32_t(acc))
      : "memory");
}
// A operand read from TMEM (M lanes x K columns, one tf32 per 32-bit column).
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(uint32_t(acc))
      : "memory");
}
// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ------------------------------------------------------------------ operand layout
// Byte offset of element (row, col) in a K-major SW128 tile with `rows` rows and elements
// of `es` bytes.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int row, int col, int rows, int es) {
  const int per_row = 128 / es;
  const int panel = col / per_row;
  const int byte = (col % per_row) * es;
  const int chunk = (byte >> 4) ^ (row & 7);
  return uint32_t(panel * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 + (chunk << 4) + (byte & 15));
}

// fp32 -> tf32, round to nearest with ties away from zero, kept in an fp32 container (the low
// 13 bits cleared). Done on the bit pattern: adding half a tf32 unit in the last place (bit 12)
// to the magnitude bits and clearing bits 0..12 rounds the magnitude to the nearest tf32 value,
// a carry out of the mantissa stepping into the exponent as rounding requires; the sign bit is
// untouched. Two integer instructions instead of the conversion instruction, which is the
// bottleneck of the conversion-heavy loops. Finite values and infinities only (a NaN whose low
// 31 bits are all set would not stay a NaN).
__device__ __forceinline__ float to_tf32(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u);
}

}  // namespace gdn
