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
// Each CTA keeps its slice of the row's keys in shared memory; per radix pass
// each CTA builds the digit histogram of its slice and every CTA merges all CS
// histograms through distributed shared memory (identical arithmetic in every
// CTA, so all reach the same digit).  The compaction writes in index order: a
// CTA's output offset is the count its lower-ranked peers select, and within a
// CTA one block scan per 1024-key chunk orders the selected keys.
__global__ void __launch_bounds__(kTopkThreads) k_topk_cluster(CacheView c, int n_q, const float *scores,
                                                               long long stride, int k, int32_t *out_idx,
                                                               int32_t *out_count, int slice_cap) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ unsigned keys[];             // [slice_cap]
  __shared__ unsigned hist[256];
  __shared__ int scan_buf[64];
  __shared__ unsigned sh_prefix;
  __shared__ int sh_krem;
  __shared__ int cnt[2];                         // this CTA's (greater, equal) counts
  __shared__ int merged[256];
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
  for (int j = threadIdx.x; j < len; j += blockDim.x) keys[j] = float_key(__ldg(s + j));
  unsigned prefix = 0, mask = 0;
  int krem = k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int e = threadIdx.x; e < 256; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < len; j += blockDim.x) {
      const unsigned key = keys[j];
      const bool in = (key & mask) == prefix;
      const unsigned bin = (key >> shift) & 255u;
      const unsigned act = __ballot_sync(__activemask(), in);
      if (in) {
        const unsigned peers = __match_any_sync(act, bin);
        if ((threadIdx.x & 31) == (unsigned)(__ffs(peers) - 1)) atomicAdd(&hist[bin], __popc(peers));
      }
    }
    cl.sync();   // every slice histogram complete and visible to the cluster
    if (threadIdx.x < 256) {
      int cdig = 0;
      for (int r = 0; r < CS; ++r) cdig += (int)cl.map_shared_rank(hist, r)[threadIdx.x];
      merged[threadIdx.x] = cdig;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l owns bins 255-8l .. 248-8l (descending); find the bin where the
      // count of larger keys reaches krem
      int part = 0;
      for (int q = 0; q < 8; ++q) part += merged[255 - 8 * threadIdx.x - q];
      int incl = part;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if ((int)threadIdx.x >= o) incl += y;
      }
      const int before = incl - part;
      if (before < krem && incl >= krem) {
        int cum = before;
        for (int q = 0; q < 8; ++q) {
          const int dgt = 255 - 8 * threadIdx.x - q;
          if (cum + merged[dgt] >= krem) {
            sh_prefix = prefix | ((unsigned)dgt << shift);
            sh_krem = krem - cum;
            break;
          }
          cum += merged[dgt];
        }
      }
    }
    cl.sync();   // peers are done reading this CTA's histogram; digit published
    prefix = sh_prefix;
    krem = sh_krem;
    mask |= 255u << shift;
  }
  // counts of this slice
  int gt = 0, eq = 0;
  for (int j = threadIdx.x; j < len; j += blockDim.x) {
    gt += keys[j] > prefix;
    eq += keys[j] == prefix;
  }
  int tg, te;
  block_exclusive_scan(gt, scan_buf, tg);
  block_exclusive_scan(eq, scan_buf, te);
  if (threadIdx.x == 0) { cnt[0] = tg; cnt[1] = te; }
  cl.sync();
  long long base = 0;
  int eq_before = 0;
  for (int r = 0; r < rank; ++r) {
    const int *pc = cl.map_shared_rank(cnt, r);
    const int g_r = pc[0], e_r = pc[1];
    base += g_r + max(0, min(e_r, krem - eq_before));
    eq_before += e_r;
  }
  int limit = max(0, krem - eq_before);   // equal keys this CTA may still take, in index order
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  for (int c0 = 0; c0 < len; c0 += blockDim.x) {
    const int j = c0 + threadIdx.x;
    const bool valid = j < len;
    const unsigned key = valid ? keys[j] : 0u;
    const bool isg = valid && key > prefix, ise = valid && key == prefix;
    const unsigned bg = __ballot_sync(0xffffffffu, isg), be = __ballot_sync(0xffffffffu, ise);
    const int packed = (int)(((unsigned)__popc(be) << 16) | (unsigned)__popc(bg));
    int tot;
    const int ex = block_exclusive_scan(lane == 0 ? packed : 0, scan_buf, tot);
    const int wex = __shfl_sync(0xffffffffu, ex, 0);
    const int G_w = wex & 0xFFFF, E_w = wex >> 16;
    const int erank = E_w + __popc(be & lt);
    const bool take = isg || (ise && erank < limit);
    const unsigned bt = __ballot_sync(0xffffffffu, take);
    if (take) {
      const long long pos = base + G_w + min(limit, E_w) + __popc(bt & lt);
      out[pos] = (int32_t)(lo + j);
    }
    const int G = tot & 0xFFFF, E = tot >> 16;
    base += G + min(limit, E);
    limit -= min(limit, E);
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
  if (smem > 160 * 1024) {
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
