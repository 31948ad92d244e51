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

// One CTA. Sequence n covers rows [cu[n], cu[n+1]) (dense: [n*T, (n+1)*T)). Sequences are
// taken in rounds of blockDim.x: a block-wide scan of their chunk counts gives each its first
// chunk, then every thread writes chunk entries of the round (chunk q of the round belongs to
// the first sequence whose inclusive count exceeds q), so a long sequence's entries are written
// by the whole block, not by one thread.
__global__ void __launch_bounds__(1024) k_tables(const TableParams p) {
  __shared__ int carry;
  __shared__ int scan[1024];
  __shared__ int s_start[1024], s_len[1024];
  const int tid = threadIdx.x, nt = blockDim.x;
  if (tid == 0) {
    carry = 0;
    if (p.status) *p.status = 0;
  }
  __syncthreads();
  for (int base = 0; base < p.N; base += nt) {
    const int n = base + tid;
    int start = 0, len = 0;
    if (n < p.N) {
      start = p.cu ? p.cu[n] : n * p.T;
      const int end = p.cu ? p.cu[n + 1] : (n + 1) * p.T;
      len = end - start;
    }
    const int nch = (len + kC - 1) / kC;
    scan[tid] = nch;
    s_start[tid] = start;
    s_len[tid] = len;
    __syncthreads();
    for (int off = 1; off < nt; off <<= 1) {  // inclusive Hillis-Steele scan
      const int add = tid >= off ? scan[tid - off] : 0;
      __syncthreads();
      scan[tid] += add;
      __syncthreads();
    }
    const int c0 = carry, total = scan[nt - 1];
    if (n < p.N) p.seqs[n] = make_int2(c0 + scan[tid] - nch, nch);
    for (int q = tid; q < total; q += nt) {
      int lo = 0, hi = nt - 1;  // first i with scan[i] > q (empty sequences are never chosen)
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (scan[mid] > q) hi = mid; else lo = mid + 1;
      }
      const int j = q - (lo > 0 ? scan[lo - 1] : 0);
      const int rows = min(kC, s_len[lo] - j * kC);
      if (c0 + q < p.NC) p.chunks[c0 + q] = make_int4(s_start[lo] + j * kC, rows, base + lo, j);
    }
    __syncthreads();
    if (tid == 0) carry += total;
    __syncthreads();
  }
}

cudaError_t launch_upload(const UploadParams& p, int* dst, cudaStream_t s) {
  k_upload<<<1, 256, 0, s>>>(p, dst);
  return cudaGetLastError();
}

cudaError_t launch_tables(const TableParams& p, cudaStream_t s) {
  // as many threads as sequences (whole warps, at least 128 to share the chunk writes, at
  // most 1024): a short scan for a small batch
  const int threads = std::min(1024, std::max(128, (p.N + 31) / 32 * 32));
  k_tables<<<1, threads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
