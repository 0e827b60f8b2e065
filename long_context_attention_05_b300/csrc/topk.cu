// a3 — top-k selection over indexer scores.
//
// Source: "DeepSeek V4: How They Crushed the Million-Token Memory Problem"
// (sameershanbhag.com), "Two kinds of memory instead of one" — the indexer keeps
// only the top-k most relevant compressed blocks for each query.
//
// Radix select on the order-preserving 32-bit image of each score: four passes of
// an 8-bit digit histogram find the exact k-th largest key T and how many of
// the entries equal to T are still needed; one compaction pass then writes, in
// ascending index order, every entry above T plus the lowest-index entries equal
// to T.  Integer counting only, so the result is deterministic and independent
// of launch shape.  One CTA per query row.
#include "kernels.h"

namespace csa {

constexpr int kTopkThreads = 1024;

__device__ __forceinline__ int block_exclusive_scan(int v, int *buf, int &total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) buf[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = lane < (int)(blockDim.x >> 5) ? buf[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    buf[32 + lane] = s;   // inclusive warp-total prefix
  }
  __syncthreads();
  total = buf[32 + (blockDim.x >> 5) - 1];
  return (w ? buf[32 + w - 1] : 0) + x - v;
}

__global__ void __launch_bounds__(kTopkThreads) k_topk_row(CacheView c, int n_q, const float *scores,
                                                           long long stride, int k, int32_t *out_idx,
                                                           int32_t *out_count) {
  __shared__ unsigned hist[256];
  __shared__ int scan_buf[64];
  __shared__ unsigned sh_prefix;
  __shared__ int sh_krem;
  const int row = blockIdx.x;
  const int b = row / n_q, i = row % n_q;
  const long long t = c.n_tokens[b] - n_q + i;
  long long n = min((t + 1) / c.m, c.cap);
  if (n > stride) n = stride;
  const float *s = scores + (long long)row * stride;
  int32_t *out = out_idx + (long long)row * k;
  if (n <= k) {
    for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = j < n ? j : -1;
    if (threadIdx.x == 0) out_count[row] = (int32_t)n;
    return;
  }
  unsigned prefix = 0, mask = 0;
  int krem = k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int e = threadIdx.x; e < 256; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    for (long long j = threadIdx.x; j < n; j += blockDim.x) {
      const unsigned key = float_key(__ldg(s + j));
      const bool in = (key & mask) == prefix;
      const unsigned bin = (key >> shift) & 255u;
      // warp-aggregated increment: lanes with the same bin add once
      const unsigned act = __ballot_sync(__activemask(), in);
      if (in) {
        const unsigned peers = __match_any_sync(act, bin);
        if ((threadIdx.x & 31) == (unsigned)(__ffs(peers) - 1)) atomicAdd(&hist[bin], __popc(peers));
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned cum = 0;
      int digit = 0;
      for (int dgt = 255; dgt >= 0; --dgt) {
        if (cum + hist[dgt] >= (unsigned)krem) { digit = dgt; break; }
        cum += hist[dgt];
      }
      sh_prefix = prefix | ((unsigned)digit << shift);
      sh_krem = krem - (int)cum;
    }
    __syncthreads();
    prefix = sh_prefix;
    krem = sh_krem;
    mask |= 255u << shift;
    __syncthreads();
  }
  // prefix = T (k-th largest key); take all keys > T and the first krem keys == T
  const long long seg = (n + blockDim.x - 1) / blockDim.x;
  const long long lo = threadIdx.x * seg, hi = min(n, lo + seg);
  int gt = 0, eq = 0;
  for (long long j = lo; j < hi; ++j) {
    const unsigned key = float_key(__ldg(s + j));
    gt += key > prefix;
    eq += key == prefix;
  }
  int tot;
  const int eq_before = block_exclusive_scan(eq, scan_buf, tot);
  const int take_eq = max(0, min(eq, krem - eq_before));
  const int pos0 = block_exclusive_scan(gt + take_eq, scan_buf, tot);
  int pos = pos0, eq_left = take_eq;
  for (long long j = lo; j < hi; ++j) {
    const unsigned key = float_key(__ldg(s + j));
    if (key > prefix || (key == prefix && eq_left > 0)) {
      if (key == prefix) --eq_left;
      out[pos++] = (int32_t)j;
    }
  }
  if (threadIdx.x == 0) out_count[row] = k;
}

cudaError_t launch_topk(const CacheView &c, int batch, int n_q, const float *scores, long long stride, int k,
                        int32_t *out_idx, int32_t *out_count, cudaStream_t st) {
  k_topk_row<<<batch * n_q, kTopkThreads, 0, st>>>(c, n_q, scores, stride, k, out_idx, out_count);
  return cudaGetLastError();
}

}  // namespace csa
