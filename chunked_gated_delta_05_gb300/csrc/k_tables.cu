// Chunk tables: map every 64-token chunk of every sequence to its token rows.
//
// Each document is chunked from its own first token (the per-document chunk list of the
// packed KDA interface, `_packed_metadata`: ceil(len/64) chunks per document, in document
// order); a document's last chunk may be partial and is masked, never padded in memory.
#include <algorithm>

#include "common.cuh"

namespace gdn {

__global__ void k_upload(const __grid_constant__ UploadParams p, int* dst) {
  for (int i = threadIdx.x; i < p.count; i += blockDim.x) dst[i] = p.vals[i];
}

// One CTA. Sequence n covers rows [cu[n], cu[n+1]) (dense: [n*T, (n+1)*T)).
__global__ void __launch_bounds__(1024) k_tables(const TableParams p) {
  __shared__ int carry;
  __shared__ int scan[1024];
  if (threadIdx.x == 0) {
    carry = 0;
    if (p.status) *p.status = 0;
  }
  __syncthreads();
  for (int base = 0; base < p.N; base += blockDim.x) {
    const int n = base + threadIdx.x;
    int start = 0, len = 0;
    if (n < p.N) {
      start = p.cu ? p.cu[n] : n * p.T;
      const int end = p.cu ? p.cu[n + 1] : (n + 1) * p.T;
      len = end - start;
    }
    const int nch = (len + kC - 1) / kC;
    scan[threadIdx.x] = nch;
    __syncthreads();
    for (int off = 1; off < blockDim.x; off <<= 1) {  // inclusive Hillis-Steele scan
      const int add = threadIdx.x >= off ? scan[threadIdx.x - off] : 0;
      __syncthreads();
      scan[threadIdx.x] += add;
      __syncthreads();
    }
    const int first = carry + scan[threadIdx.x] - nch;
    if (n < p.N) {
      p.seqs[n] = make_int2(first, nch);
      for (int j = 0; j < nch; ++j) {
        const int rows = min(kC, len - j * kC);
        if (first + j < p.NC) p.chunks[first + j] = make_int4(start + j * kC, rows, n, j);
      }
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry += scan[threadIdx.x];
    __syncthreads();
  }
}

cudaError_t launch_upload(const UploadParams& p, int* dst, cudaStream_t s) {
  k_upload<<<1, 256, 0, s>>>(p, dst);
  return cudaGetLastError();
}

cudaError_t launch_tables(const TableParams& p, cudaStream_t s) {
  // as many threads as sequences (whole warps, at most 1024): a short scan for a small batch
  const int threads = std::min(1024, std::max(32, (p.N + 31) / 32 * 32));
  k_tables<<<1, threads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
