// Allocation-free forward: gdn_fwd with its workspace taken from a fixed static device array.
//
// Some callers cannot call cudaMalloc at the point where they run the layer: code executing
// inside an allocator-restricted region (a CUDA graph being captured, where allocation calls
// are illegal), embedders whose memory is owned by a framework allocator that must not be
// bypassed, and real-time paths that forbid allocation for latency reasons. For them this
// file provides gdn_fwd_noalloc(), which runs exactly the same kernels as gdn_fwd() but uses
// g_gdn_fwd_scratch below as its workspace. It calls no cudaMalloc / cudaFree and no other
// allocating routine.
//
// Limits and sharing:
//  * The scratch array is kNoAllocScratchBytes (32 MiB). Every GPU that loads this library
//    holds that much device memory until the process exits. Problems whose forward workspace
//    (gdn_fwd_workspace_size) is larger are rejected with GDN_EINVAL.
//  * All calls on a device share the one array, and it keeps the previous call's contents.
//    Every region the forward reads is written earlier in the same call, so nothing needs
//    clearing between calls; but two calls whose work overlaps on the GPU (different streams,
//    or host threads) race on the array and corrupt each other's results.
//  * Host code cannot use the array's name as a device address. The first call on each
//    device, with that device current, looks the address up with cudaGetSymbolAddress and
//    caches it. Make that first call before any stream capture begins.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "gdn.h"

namespace gdn {
int set_last_error(int code, const char* msg);
}

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_gdn_fwd_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

}  // namespace

extern "C" size_t gdn_fwd_noalloc_capacity(void) { return kNoAllocScratchBytes; }

extern "C" int gdn_fwd_noalloc(const gdn_desc_t* desc, const gdn_fwd_args_t* args, void* stream) {
  if (!args) return gdn_fwd(desc, args, stream);  // reports the NULL-args contract error
  if (args->workspace || args->workspace_bytes || args->saved || args->saved_bytes)
    return gdn::set_last_error(GDN_EINVAL, "gdn_fwd_noalloc takes no workspace or saved buffer: pass NULL and 0");
  const size_t need = gdn_fwd_workspace_size(desc);
  if (need == 0) return gdn_fwd(desc, args, stream);  // reports the description error
  if (need > kNoAllocScratchBytes) {
    char msg[160];
    snprintf(msg, sizeof(msg), "problem needs %zu bytes of forward workspace; gdn_fwd_noalloc has %zu (32 MiB)",
             need, kNoAllocScratchBytes);
    return gdn::set_last_error(GDN_EINVAL, msg);
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return gdn::set_last_error(GDN_EUNSUPPORTED, "no usable current CUDA device");
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_gdn_fwd_scratch) != cudaSuccess || !p)
        return gdn::set_last_error(GDN_ECUDA, "cudaGetSymbolAddress of the static scratch array failed");
      g_addr[dev] = p;
    }
    base = g_addr[dev];
  }
  gdn_fwd_args_t a = *args;
  a.workspace = base;
  a.workspace_bytes = kNoAllocScratchBytes;
  return gdn_fwd(desc, &a, stream);
}
