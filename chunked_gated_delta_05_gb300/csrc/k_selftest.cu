// Self-test of the bounded device wait that every kernel of the library uses (umma.cuh
// mbar_wait): a wait whose barrier nothing will ever complete must give up after its limit,
// record the timeout in the caller's status word and let the CTA wind down without trapping,
// so the context stays usable.
//
// One CTA of four warps. It takes TMEM columns and starts one bulk copy into shared memory
// (which completes), then every thread waits, with the caller's short limit, on a barrier that
// no thread or copy arrives on. The first thread past the limit records kDevTimeoutSync and
// raises the CTA's abort flag; the other threads see the flag and leave their waits. Before
// freeing anything the abort path waits, with the normal limit, for the copy still in flight,
// then releases TMEM and exits.
#include "common.cuh"
#include "gdn.h"
#include "umma.cuh"

namespace gdn {

namespace {
constexpr uint32_t kProbeBytes = 4096;
}

__global__ void __launch_bounds__(128) k_wait_probe(const uint8_t* src, int* status, unsigned long long limit_ns) {
  __shared__ alignas(128) uint8_t buf[kProbeBytes];
  __shared__ uint64_t bar_copy, bar_never;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) tmem_alloc(&tslot, 32);
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar_copy, 1);
    mbar_init(&bar_never, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    mbar_expect_tx(&bar_copy, kProbeBytes);
    bulk_load(buf, src, kProbeBytes, &bar_copy);
  }
  // the wait under test: bar_never's phase 0 never completes
  mbar_wait(&bar_never, 0, &abort_flag, status, kDevTimeoutSync, limit_ns);
  // abort path: the copy in flight lands before its destination is released
  if (tid == 0 && !mbar_drain(&bar_copy, 0) && status) atomicCAS(status, 0, kDevTimeoutTma);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tslot, 32);
}

}  // namespace gdn

extern "C" int gdn_wait_selftest(const void* src, long long limit_ns, int* status, void* stream) {
  if (!src || (reinterpret_cast<uintptr_t>(src) & 15) || !status || limit_ns <= 0 || limit_ns > 2000000000ll)
    return gdn::set_last_error(GDN_EINVAL, "gdn_wait_selftest: src (16-byte aligned, 4096 bytes) and status "
                                           "are required and 0 < limit_ns <= 2e9");
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return gdn::set_last_error(GDN_EUNSUPPORTED, "no CUDA device");
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return gdn::set_last_error(GDN_EUNSUPPORTED, "device is not compute capability 10.3");
  gdn::k_wait_probe<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<const uint8_t*>(src), status,
                                                                    static_cast<unsigned long long>(limit_ns));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return gdn::set_last_error(GDN_ECUDA, cudaGetErrorString(e));
  return GDN_OK;
}
