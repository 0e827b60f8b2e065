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
#include <cooperative_groups.h>

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

// Cluster version: the CS CTAs of one thread-block cluster share a query row.
// Each CTA keeps its slice of the row's keys in shared memory.  Three radix
// passes (11, 11 and 10 bits): each CTA builds the digit histogram of its
// slice; the cluster reduces it (CTA r sums bins of its own range over all
// peers) and gathers the merged histogram back through distributed shared
// memory, so every CTA holds the same histogram and reaches the same digit.
// Histograms are double-buffered across passes, so a pass costs two cluster
// barriers.  The compaction writes in index order: a CTA's output offset is
// what its lower-ranked peers select; within a CTA each thread owns a
// contiguous run of keys and one block scan orders them.
constexpr int kBins = 2048;

__global__ void __launch_bounds__(kTopkThreads) k_topk_cluster(CacheView c, int n_q, const float *scores,
                                                               long long stride, int k, int32_t *out_idx,
                                                               int32_t *out_count, int slice_cap) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ unsigned keys[];             // [slice_cap]
  __shared__ unsigned hist[2][kBins];            // this CTA's slice histogram (double-buffered)
  __shared__ unsigned part[2][kBins];            // merged counts of this CTA's bin range
  __shared__ int scan_buf[64];
  __shared__ unsigned sh_prefix;
  __shared__ int sh_krem;
  __shared__ int cnt[2];                         // this CTA's (greater, equal) counts
  const int CS = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const int row = blockIdx.y;
  const int b = row / n_q, i = row % n_q;
  const long long t = c.n_tokens[b] - n_q + i;
  long long n = min((t + 1) / c.m, c.cap);
  if (n > stride) n = stride;
  int32_t *out = out_idx + (long long)row * k;
  if (n <= k) {   // uniform over the cluster: no cluster barrier is reached
    if (rank == 0) {
      for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = j < n ? j : -1;
      if (threadIdx.x == 0) out_count[row] = (int32_t)n;
    }
    return;
  }
  const long long L = (n + CS - 1) / CS;
  const long long lo = min(n, rank * L), hi = min(n, lo + L);
  const int len = (int)(hi - lo);
  const float *s = scores + (long long)row * stride + lo;
  // eight loads in flight per thread per round (not one memory round trip per key)
  for (int j0 = 0; j0 < len; j0 += 8 * kTopkThreads) {
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = j0 + q * kTopkThreads + (int)threadIdx.x;
      v[q] = j < len ? __ldg(s + j) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = j0 + q * kTopkThreads + (int)threadIdx.x;
      if (j < len) keys[j] = float_key(v[q]);
    }
  }
  const int per = kBins / CS;                    // bins this CTA reduces
  unsigned prefix = 0, mask = 0;
  int krem = k;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass];
    const unsigned dmask = (1u << widths[pass]) - 1u;
    unsigned *h = hist[pass & 1];
    unsigned *pm = part[pass & 1];
    for (int e = threadIdx.x; e < kBins; e += blockDim.x) h[e] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < len; j += blockDim.x) {
      const unsigned key = keys[j];
      const bool in = (key & mask) == prefix;
      const unsigned bin = (key >> shift) & dmask;
      const unsigned act = __ballot_sync(__activemask(), in);
      if (in) {
        const unsigned peers = __match_any_sync(act, bin);
        if ((threadIdx.x & 31) == (unsigned)(__ffs(peers) - 1)) atomicAdd(&h[bin], __popc(peers));
      }
    }
    cl.sync();   // all slice histograms complete
    for (int e = threadIdx.x; e < per; e += blockDim.x) {
      unsigned v[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) v[r] = r < CS ? cl.map_shared_rank(h, r)[rank * per + e] : 0u;   // all in flight
      unsigned sum = 0;
#pragma unroll
      for (int r = 0; r < 16; ++r) sum += v[r];
      pm[rank * per + e] = sum;
    }
    cl.sync();   // every CTA's merged range complete
    // gather the merged histogram; thread x owns bins 2047-2x and 2046-2x (descending)
    const int b0 = kBins - 1 - 2 * (int)threadIdx.x, b1 = b0 - 1;
    const unsigned c0 = cl.map_shared_rank(pm, b0 / per)[b0];
    const unsigned c1 = cl.map_shared_rank(pm, b1 / per)[b1];
    int tot;
    const int above = block_exclusive_scan((int)(c0 + c1), scan_buf, tot);   // keys in higher bins
    if (above < krem && above + (int)(c0 + c1) >= krem) {
      const bool first = above + (int)c0 >= krem;
      sh_prefix = prefix | ((unsigned)(first ? b0 : b1) << shift);
      sh_krem = krem - (first ? above : above + (int)c0);
    }
    __syncthreads();
    prefix = sh_prefix;
    krem = sh_krem;
    mask |= dmask << shift;
  }
  // prefix = T, the k-th largest key; krem keys equal to T are still to be taken.
  // Warp w owns the contiguous run [w*seg, (w+1)*seg) of this slice and walks it
  // 32 keys at a time (coalesced, conflict-free); ballots order keys inside a
  // round, one block scan orders the warps.
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = (int)blockDim.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const int seg = ((len + nwarps - 1) / nwarps + 31) & ~31;
  const int w0 = min(len, warp * seg), w1 = min(len, w0 + seg);
  int gw = 0, ew = 0;   // this warp's counts of keys > T and == T
  for (int j0 = w0; j0 < w1; j0 += 32) {
    const int j = j0 + lane;
    const unsigned key = j < w1 ? keys[j] : 0u;
    gw += __popc(__ballot_sync(0xffffffffu, j < w1 && key > prefix));
    ew += __popc(__ballot_sync(0xffffffffu, j < w1 && key == prefix));
  }
  int tot;
  const int ex = block_exclusive_scan(lane == 0 ? ((ew << 16) | gw) : 0, scan_buf, tot);   // counts < 2^16
  const int wex = __shfl_sync(0xffffffffu, ex, 0);
  if (threadIdx.x == 0) { cnt[0] = tot & 0xFFFF; cnt[1] = tot >> 16; }
  cl.sync();
  long long base = 0;
  int eq_before = 0;
  int pg[16], pe[16];
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    pg[r] = r < rank ? cl.map_shared_rank(cnt, r)[0] : 0;
    pe[r] = r < rank ? cl.map_shared_rank(cnt, r)[1] : 0;
  }
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    base += pg[r] + max(0, min(pe[r], krem - eq_before));
    eq_before += pe[r];
  }
  const int limit = max(0, krem - eq_before);   // equal keys this CTA may take, in index order
  int e_seen = wex >> 16;                        // equal keys before this warp's run (in this CTA)
  long long pos = base + (wex & 0xFFFF) + min(limit, e_seen);
  for (int j0 = w0; j0 < w1; j0 += 32) {
    const int j = j0 + lane;
    const unsigned key = j < w1 ? keys[j] : 0u;
    const bool isg = j < w1 && key > prefix, ise = j < w1 && key == prefix;
    const unsigned be = __ballot_sync(0xffffffffu, ise);
    const bool take = isg || (ise && e_seen + __popc(be & lt) < limit);
    const unsigned bt = __ballot_sync(0xffffffffu, take);
    if (take) out[pos + __popc(bt & lt)] = (int32_t)(lo + j);
    pos += __popc(bt);
    e_seen += __popc(be);
  }
  if (rank == 0 && threadIdx.x == 0) out_count[row] = k;
  cl.sync();   // no CTA leaves while a peer may still read its shared memory
}

// Rows with few queries get a cluster of up to 16 CTAs each; many rows get one
// CTA each.  Rows whose slice would not fit in shared memory use k_topk_row.
cudaError_t launch_topk(const CacheView &c, int batch, int n_q, const float *scores, long long stride, int k,
                        int32_t *out_idx, int32_t *out_count, int num_sms, cudaStream_t st) {
  const int rows = batch * n_q;
  const long long n_cap = c.cap < stride ? c.cap : stride;
  int cs = 1;
  if (rows < num_sms) {
    cs = 16;
    while (cs > 1 && (long long)rows * cs > 2LL * num_sms && (n_cap + cs / 2 - 1) / (cs / 2) <= 32768) cs /= 2;
  }
  const long long slice = (n_cap + cs - 1) / cs;
  const size_t smem = (size_t)slice * sizeof(unsigned);
  if (smem > 160 * 1024 || cs > 16 || kBins % cs) {
    k_topk_row<<<rows, kTopkThreads, 0, st>>>(c, n_q, scores, stride, k, out_idx, out_count);
    return cudaGetLastError();
  }
  cudaError_t e = cudaFuncSetAttribute(k_topk_cluster, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess && cs > 8)
    e = cudaFuncSetAttribute(k_topk_cluster, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  for (;; cs /= 2) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, rows);
    cfg.blockDim = dim3(kTopkThreads);
    cfg.dynamicSmemBytes = (size_t)((n_cap + cs - 1) / cs) * sizeof(unsigned);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cfg.dynamicSmemBytes > 160 * 1024) break;
    e = cudaLaunchKernelEx(&cfg, k_topk_cluster, c, n_q, scores, stride, k, out_idx, out_count,
                           (int)((n_cap + cs - 1) / cs));
    if (e == cudaSuccess || cs == 1) return e;
    cudaGetLastError();   // cluster too large for this device: halve it
  }
  k_topk_row<<<rows, kTopkThreads, 0, st>>>(c, n_q, scores, stride, k, out_idx, out_count);
  return cudaGetLastError();
}

}  // namespace csa
