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
// the row-split kernel's last CTA holds the row's list (fewer than k + kCandMax
// entries) in registers, this many per thread: the kernel serves k + kCandMax <=
// kSplitRun * kTopkThreads
constexpr int kSplitRun = 8;

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

// block_exclusive_scan for two counts at once (one set of barriers)
__device__ __forceinline__ int2 block_exclusive_scan2(int2 v, int2 *buf, int2 &total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int2 x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int yx = __shfl_up_sync(0xffffffffu, x.x, o), yy = __shfl_up_sync(0xffffffffu, x.y, o);
    if (lane >= o) { x.x += yx; x.y += yy; }
  }
  __syncthreads();
  if (lane == 31) buf[w] = x;
  __syncthreads();
  if (w == 0) {
    int2 s = lane < (int)(blockDim.x >> 5) ? buf[lane] : make_int2(0, 0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yx = __shfl_up_sync(0xffffffffu, s.x, o), yy = __shfl_up_sync(0xffffffffu, s.y, o);
      if (lane >= o) { s.x += yx; s.y += yy; }
    }
    buf[32 + lane] = s;   // inclusive warp-total prefix
  }
  __syncthreads();
  total = buf[32 + (blockDim.x >> 5) - 1];
  const int2 before = w ? buf[32 + w - 1] : make_int2(0, 0);
  return make_int2(before.x + x.x - v.x, before.y + x.y - v.y);
}

// A nonzero status word (the indexer's bounded wait gave up, so the scores are
// incomplete): the row gets count -1 and all-(-1) indices instead of a selection.
__device__ __forceinline__ bool status_failed(const int *status) {
  return status != nullptr && *reinterpret_cast<const volatile int *>(status) != 0;
}

// Single-CTA radix select over one row's n > k scores s (k_topk_row with
// kRowThreads, the row-split kernel's fallback with kTopkThreads; any block of
// 256..1024 threads that divides 2048): three passes of an 11-,
// 11- and 10-bit digit histogram find T, the k-th largest key, and how many keys
// equal to T to take; one count pass and one write pass then emit the selection in
// index order.  The histogram passes stream the row as 16-byte loads, 16 keys per
// thread in flight (the passes are bound by load latency, not by arithmetic).
__device__ void radix_select_row(const float *s, long long n, int k, int32_t *out) {
  constexpr int kRB = 2048;   // digit bins
  __shared__ unsigned hist[kRB];
  __shared__ int scan_buf[64];
  __shared__ int2 scan_buf2[64];
  __shared__ unsigned sh_prefix;
  __shared__ int sh_krem;
  const int lane = threadIdx.x & 31;
  // [0, head) and [tail0, n) as scalars, the 16-byte aligned middle as float4s
  const int head = (int)min(n, (long long)((4 - (((uintptr_t)s >> 2) & 3)) & 3));
  const long long nvec = (n - head) >> 2;
  const long long tail0 = head + 4 * nvec;
  const float4 *sv = reinterpret_cast<const float4 *>(s + head);
  unsigned prefix = 0, mask = 0;
  int krem = k;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : pass == 1 ? 10 : 0;
    const unsigned dmask = pass == 2 ? 0x3FFu : 0x7FFu;
    for (int e = threadIdx.x; e < kRB; e += blockDim.x) hist[e] = 0u;
    __syncthreads();
    // one key per lane, counted once per distinct bin in the warp (rows with few
    // distinct keys would otherwise serialise up to 32 atomics on one word); a warp
    // whose keys all fall in one bin adds 32 to a count it holds in registers while
    // the bin repeats (rows of equal keys: one atomic per warp and pass)
    unsigned run_bin = 0u, run_cnt = 0u;   // warp-uniform
    auto add = [&](unsigned key, bool valid) {
      const bool in = valid && (key & mask) == prefix;
      const unsigned bin = (key >> shift) & dmask;
      const unsigned b0 = __shfl_sync(0xffffffffu, bin, 0);
      if (__all_sync(0xffffffffu, in && bin == b0)) {
        if (run_cnt && b0 != run_bin) {
          if (lane == 0) atomicAdd(&hist[run_bin], run_cnt);
          run_cnt = 0u;
        }
        run_bin = b0;
        run_cnt += 32u;
        return;
      }
      const unsigned act = __ballot_sync(0xffffffffu, in);
      if (in) {
        const unsigned peers = __match_any_sync(act, bin);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist[bin], (unsigned)__popc(peers));
      }
    };
    for (long long v0 = 0; v0 < nvec; v0 += 4LL * blockDim.x) {   // the same trip count in every thread
      float4 f[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const long long x = v0 + (long long)q * blockDim.x + threadIdx.x;
        f[q] = x < nvec ? __ldg(sv + x) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const bool valid = v0 + (long long)q * blockDim.x + threadIdx.x < nvec;
        add(float_key(f[q].x), valid);
        add(float_key(f[q].y), valid);
        add(float_key(f[q].z), valid);
        add(float_key(f[q].w), valid);
      }
    }
    if (threadIdx.x < 32) {   // the at most 3 + 3 unaligned keys at the ends
      const long long j = lane < head ? lane : tail0 + (lane - head);
      const bool valid = lane < head || (j >= tail0 && j < n);
      add(valid ? float_key(__ldg(s + j)) : 0u, valid);
    }
    if (lane == 0 && run_cnt) atomicAdd(&hist[run_bin], run_cnt);
    __syncthreads();
    // the digit of T: thread x owns the bpt bins from 2047 - bpt x down (descending)
    const int bpt = kRB / (int)blockDim.x;
    const int top = kRB - 1 - bpt * (int)threadIdx.x;
    int csum = 0;
    for (int q = 0; q < bpt; ++q) csum += (int)hist[top - q];
    int tot;
    const int above = block_exclusive_scan(csum, scan_buf, tot);
    if (above < krem && above + csum >= krem) {
      int cum = above;
      for (int q = 0; q < bpt; ++q) {
        const int cq = (int)hist[top - q];
        if (cum + cq >= krem) {
          sh_prefix = prefix | ((unsigned)(top - q) << shift);
          sh_krem = krem - cum;
          break;
        }
        cum += cq;
      }
    }
    __syncthreads();
    prefix = sh_prefix;
    krem = sh_krem;
    mask |= dmask << shift;
  }
  // prefix = T; take all keys > T and the first krem keys == T, in index order.  One
  // coalesced pass in rounds of 8 keys per thread (key base + q * blockDim.x + x in
  // thread x: index order is (q, warp, lane)); ballots rank a key inside its warp, one
  // block scan of the (q, warp) counts ranks the warps, running totals rank the rounds;
  // the next round's keys load while this round is ranked.  A taken key's position is
  // (keys > T before it) + min(keys == T before it, krem).
  {
    constexpr int kQ = 8;
    __shared__ int2 wc[kQ * 32];
    const int warp = threadIdx.x >> 5, nwarps = (int)blockDim.x >> 5;
    const unsigned lt = (1u << lane) - 1u;
    const long long step = (long long)kQ * blockDim.x;
    long long run_gt = 0, run_eq = 0;   // keys > T and == T in earlier rounds (uniform)
    unsigned nk[kQ];
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      const long long j = (long long)q * blockDim.x + threadIdx.x;
      nk[q] = j < n ? float_key(__ldg(s + j)) : 0u;
    }
    for (long long base = 0; base < n && run_gt + min(run_eq, (long long)krem) < k; base += step) {
      unsigned kq[kQ], bg[kQ], be[kQ];
#pragma unroll
      for (int q = 0; q < kQ; ++q) kq[q] = nk[q];
#pragma unroll
      for (int q = 0; q < kQ; ++q) {   // the next round's keys
        const long long j = base + step + (long long)q * blockDim.x + threadIdx.x;
        nk[q] = j < n ? float_key(__ldg(s + j)) : 0u;
      }
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const bool valid = base + (long long)q * blockDim.x + threadIdx.x < n;
        bg[q] = __ballot_sync(0xffffffffu, valid && kq[q] > prefix);
        be[q] = __ballot_sync(0xffffffffu, valid && kq[q] == prefix);
        if (lane == 0) wc[q * nwarps + warp] = make_int2(__popc(bg[q]), __popc(be[q]));
      }
      __syncthreads();
      const int2 v = (int)threadIdx.x < kQ * nwarps ? wc[threadIdx.x] : make_int2(0, 0);
      int2 tot;
      const int2 ex = block_exclusive_scan2(v, scan_buf2, tot);
      if ((int)threadIdx.x < kQ * nwarps) wc[threadIdx.x] = ex;
      __syncthreads();
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const int2 o = wc[q * nwarps + warp];
        const long long gb = run_gt + o.x + __popc(bg[q] & lt), eb = run_eq + o.y + __popc(be[q] & lt);
        const long long j = base + (long long)q * blockDim.x + threadIdx.x;
        if ((bg[q] >> lane) & 1u) out[gb + min(eb, (long long)krem)] = (int32_t)j;
        else if (((be[q] >> lane) & 1u) && eb < krem) out[gb + eb] = (int32_t)j;
      }
      run_gt += tot.x;
      run_eq += tot.y;
      __syncthreads();   // wc is rewritten by the next round
    }
  }
}

// One query row per CTA of kRowThreads: several CTAs share an SM, so the rows'
// load latencies overlap (the select is bound by them, not by arithmetic).
constexpr int kRowThreads = 256;

__global__ void __launch_bounds__(kRowThreads) k_topk_row(CacheView c, int n_q, const float *scores,
                                                           long long stride, int k, int32_t *out_idx,
                                                           int32_t *out_count, const int *status) {
  const int row = blockIdx.x;
  const int b = row / n_q, i = row % n_q;
  pdl_wait();
  pdl_trigger();
  const long long t = c.n_tokens[b] - n_q + i;
  long long n = min((t + 1) / c.m, c.cap);
  if (n > stride) n = stride;
  int32_t *out = out_idx + (long long)row * k;
  const bool failed = status_failed(status);
  if (n <= k || failed) {
    for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = (j < n && !failed) ? j : -1;
    if (threadIdx.x == 0) out_count[row] = failed ? -1 : (int32_t)n;
    return;
  }
  radix_select_row(scores + (long long)row * stride, n, k, out);
  if (threadIdx.x == 0) out_count[row] = k;
}

// Cluster version: the CS CTAs of one thread-block cluster share a query row;
// each keeps its slice of the row's keys in shared memory.
//   1. cluster-wide min and max of the scores;
//   2. one histogram over 2048 equal-width VALUE bins of [min, max] (monotone:
//      a key in a higher bin is larger than every key in a lower one), merged
//      across the cluster through distributed shared memory (CTA r sums its own
//      bin range over all peers, then every CTA gathers the merged counts);
//   3. the bin holding the k-th largest score is found by a scan from the top;
//      the few keys of that bin are gathered from all peers and the exact k-th
//      key T is found among them by rank counting;
//   4. compaction in index order: keys > T, then keys == T lowest index first.
// Bins that are too crowded (degenerate value ranges) fall back to three radix
// passes over the ordered-integer keys.  Every decision is integer counting on
// identical data in every CTA, so the result is deterministic.
// With the indexer's per-row prefix histogram (fused call), steps 1-3 start from it:
// every CTA finds the threshold prefix bin and the count above it by itself, lists
// its keys in and above that bin, and one cluster barrier later gathers all CTAs'
// keys of the bin; the histogram is checked against the keys and zeroed for the
// next call.
constexpr int kBins = 2048;

__device__ __forceinline__ float key_float(unsigned key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

__global__ void __launch_bounds__(kTopkThreads) k_topk_cluster(CacheView c, int n_q, const float *scores,
                                                               long long stride, int k, int32_t *out_idx,
                                                               int32_t *out_count, unsigned *ghist, int slice_cap,
                                                               const int *status) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ unsigned keys[];             // [slice_cap] keys, then [slice_cap] uint16 bins
  unsigned short *kbin = reinterpret_cast<unsigned short *>(keys + slice_cap);
  __shared__ unsigned hist[4][kBins];            // this CTA's slice histogram, four sub-copies
  __shared__ unsigned part[kBins];               // merged counts of this CTA's bin range
  __shared__ unsigned cand[kCandMax];            // rank 0: every CTA's candidates; then a private copy
  __shared__ unsigned char cand_rank[kCandMax];  // ... and the rank each came from
  __shared__ int above_r[16];                    // rank 0: each CTA's count of keys above the bin
  __shared__ int gt_r[16], eq_r[16];             // per rank: keys > T, keys == T
  __shared__ int scan_buf[64];
  __shared__ unsigned red_u[64];
  __shared__ unsigned sh_minmax[2];              // this CTA's (min, max) key
  __shared__ int sh_cand;                        // rank 0: candidates appended so far
  __shared__ unsigned sh_prefix;
  __shared__ int sh_krem, sh_bin, sh_above, sh_incount;
  __shared__ int cnt[2];                         // this CTA's (greater, equal) counts
  __shared__ int sh_myab;                        // fast path: this CTA's keys above the threshold bin
  const int CS = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const int row = blockIdx.y;
  const int b = row / n_q, i = row % n_q;
  pdl_wait();
  pdl_trigger();
  const long long t = c.n_tokens[b] - n_q + i;
  long long n = min((t + 1) / c.m, c.cap);
  if (n > stride) n = stride;
  int32_t *out = out_idx + (long long)row * k;
  const bool failed = status_failed(status);   // the same word for every CTA of the cluster
  if (n <= k || failed) {   // uniform over the cluster: no cluster barrier is reached
    if (rank == 0) {
      for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = (j < n && !failed) ? j : -1;
      if (threadIdx.x == 0) out_count[row] = failed ? -1 : (int32_t)n;
    }
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = (int)blockDim.x >> 5;
  const long long L = (n + CS - 1) / CS;
  const long long lo = min(n, rank * L), hi = min(n, lo + L);
  const int len = (int)(hi - lo);
  const float *s = scores + (long long)row * stride + lo;
  // the row's prefix counts (fast path, below) are loaded along with the scores
  static_assert(kPrefixBins == 8 * kTopkThreads, "one thread per 8 prefix bins");
  const int hb = kPrefixBins - 8 * ((int)threadIdx.x + 1);   // this thread's bins hb .. hb+7
  uint4 h0 = make_uint4(0, 0, 0, 0), h1 = make_uint4(0, 0, 0, 0);
  if (ghist != nullptr) {
    const unsigned *hr = ghist + (long long)row * kPrefixBins;
    h0 = *reinterpret_cast<const uint4 *>(hr + hb);
    h1 = *reinterpret_cast<const uint4 *>(hr + hb + 4);
  }
  // ---- load: 16-byte loads for the aligned middle, scalars for the ends; and the
  //      slice's min / max key
  unsigned kmin = 0xFFFFFFFFu, kmax = 0u;
  {
    const int head = min(len, (int)((4 - (((uintptr_t)s >> 2) & 3)) & 3));
    const int nvec = (len - head) >> 2;
    const float4 *sv = reinterpret_cast<const float4 *>(s + head);
    for (int v0 = 0; v0 < nvec; v0 += 4 * kTopkThreads) {
      float4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int x = v0 + q * kTopkThreads + (int)threadIdx.x;
        v[q] = x < nvec ? __ldg(sv + x) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int x = v0 + q * kTopkThreads + (int)threadIdx.x;
        if (x < nvec) {
          const unsigned k0 = float_key(v[q].x), k1 = float_key(v[q].y), k2 = float_key(v[q].z), k3 = float_key(v[q].w);
          unsigned *kd = keys + head + 4 * x;   // not 16-byte aligned in general: scalar stores
          kd[0] = k0; kd[1] = k1; kd[2] = k2; kd[3] = k3;
          kmin = min(min(kmin, min(k0, k1)), min(k2, k3));
          kmax = max(max(kmax, max(k0, k1)), max(k2, k3));
        }
      }
    }
    for (int j = threadIdx.x; j < len; j += blockDim.x) {   // the unaligned ends
      if (j < head || j >= head + 4 * nvec) {
        const unsigned key = float_key(__ldg(s + j));
        keys[j] = key;
        kmin = min(kmin, key);
        kmax = max(kmax, key);
      }
    }
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) { red_u[warp] = kmin; red_u[32 + warp] = kmax; }
  for (int e = threadIdx.x; e < kBins; e += blockDim.x) {
    hist[0][e] = 0; hist[1][e] = 0; hist[2][e] = 0; hist[3][e] = 0;
    part[e] = 0;
  }
  if (threadIdx.x < 16) { gt_r[threadIdx.x] = 0; eq_r[threadIdx.x] = 0; }
  if (threadIdx.x == 0) sh_cand = 0;
  __syncthreads();
  if (warp == 0) {
    unsigned a = lane < nwarps ? red_u[lane] : 0xFFFFFFFFu, z = lane < nwarps ? red_u[32 + lane] : 0u;
    a = __reduce_min_sync(0xffffffffu, a);
    z = __reduce_max_sync(0xffffffffu, z);
    if (lane == 0) { sh_minmax[0] = a; sh_minmax[1] = z; }
  }
  // ---- fast path: the indexer left this row's histogram of 13-bit key prefixes (bins
  //      of 1/16 octave).  If it counts exactly this row's n scores, the bin of the
  //      k-th largest key and the count above it come straight from it: no min / max,
  //      no histogram pass, no cluster exchange of histograms.
  bool fast = false;
  if (ghist != nullptr) {   // uniform
    const unsigned cb[8] = {h1.w, h1.z, h1.y, h1.x, h0.w, h0.z, h0.y, h0.x};   // descending bins
    int s8 = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) s8 += (int)cb[q];
    int tot;
    const int above = block_exclusive_scan(s8, scan_buf, tot);   // keys in higher bins
    if ((long long)tot == n && above < k && above + s8 >= k) {
      int cum = above;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (cum < k && cum + (int)cb[q] >= k) { sh_bin = hb + 7 - q; sh_above = cum; sh_incount = (int)cb[q]; }
        cum += (int)cb[q];
      }
    }
    fast = (long long)tot == n;   // the same in every thread and every CTA of the row
    __syncthreads();
  }
  unsigned prefix = 0;
  int krem = k;
  bool need_radix = false;
  bool fast_offsets = false;   // output offsets known from the candidate lists (no count exchange)
  bool fast_list = false;      // this warp's keys in or above the threshold bin are listed in kbin
  int nsel = 0;                // ... that many
  // Warp w owns the contiguous run [w*seg, (w+1)*seg) of this slice in the passes
  // below that must keep index order; it walks it 32 keys at a time (coalesced,
  // conflict-free) and ballots order the keys inside a round.
  const unsigned lt = (1u << lane) - 1u;
  const int seg = ((len + nwarps - 1) / nwarps + 31) & ~31;
  const int w0 = min(len, warp * seg), w1 = min(len, w0 + seg);
  // exact k-th key T among the threshold bin's candidates ck[0, total) (rank cr[x]
  // each), and per rank the candidates above T and equal to T
  // (pre0, msk0): bits every candidate shares; the radix passes cover the rest
  auto select_among = [&](const unsigned *ck, const unsigned char *cr, int total, int kin, unsigned pre0,
                          unsigned msk0) {
    if (total <= 128) {
      // exact rank of each candidate among the candidates
      if ((int)threadIdx.x < total) {
        const unsigned key = ck[threadIdx.x];
        int gtc = 0, eqc = 0;
        for (int y = 0; y < total; ++y) {
          gtc += ck[y] > key;
          eqc += ck[y] == key;
        }
        if (gtc < kin && gtc + eqc >= kin) {   // several equal keys write the same values
          sh_prefix = key;
          sh_krem = kin - gtc;
        }
      }
      __syncthreads();
      prefix = sh_prefix;
      krem = sh_krem;
    } else {
      // three radix passes over the candidates, inside this CTA (no cluster barrier)
      unsigned pre = pre0, msk = msk0;
      int kr = kin;
      // 11-bit digits from the top of the bits not yet fixed (the last digit may be shorter)
      const int free_bits = 32 - __popc(msk0);
      for (int hi = free_bits; hi > 0; hi -= 11) {
        const int width = hi < 11 ? hi : 11, shift = hi - width;
        const unsigned dmask = (1u << width) - 1u;
        for (int e = threadIdx.x; e < kBins; e += blockDim.x) hist[0][e] = 0;
        __syncthreads();
        for (int x = threadIdx.x; x < total; x += blockDim.x) {
          const unsigned key = ck[x];
          if ((key & msk) == pre) atomicAdd(&hist[0][(key >> shift) & dmask], 1u);
        }
        __syncthreads();
        const int b0 = kBins - 1 - 2 * (int)threadIdx.x, b1 = b0 - 1;
        const unsigned c0 = hist[0][b0], c1 = hist[0][b1];
        int tot2;
        const int above2 = block_exclusive_scan((int)(c0 + c1), scan_buf, tot2);
        if (above2 < kr && above2 + (int)(c0 + c1) >= kr) {
          const bool first = above2 + (int)c0 >= kr;
          sh_prefix = pre | ((unsigned)(first ? b0 : b1) << shift);
          sh_krem = kr - (first ? above2 : above2 + (int)c0);
        }
        __syncthreads();
        pre = sh_prefix;
        kr = sh_krem;
        msk |= dmask << shift;
      }
      prefix = pre;
      krem = kr;
    }
    // per rank: keys > T (above the bin, or candidates above T) and keys == T
    for (int x = threadIdx.x; x < total; x += blockDim.x) {
      if (ck[x] > prefix) atomicAdd(&gt_r[cr[x]], 1);
      else if (ck[x] == prefix) atomicAdd(&eq_r[cr[x]], 1);
    }
    __syncthreads();
  };
  if (fast) {
    // ---- the threshold prefix bin b* and the count above it come from the indexer's
    //      histogram.  Each CTA lists its own keys in b* and counts its keys above b*;
    //      after one cluster barrier every CTA gathers all lists.  A histogram that
    //      does not match the keys (lists or counts differ from it) falls back to the
    //      radix passes, so a stale histogram costs time, never correctness.
    const unsigned bstar = (unsigned)sh_bin;
    const int kin = k - sh_above, total = sh_incount;
    bool ok = total <= kCandMax;   // uniform
    if (ok) {
      // warp runs as in the output passes below: each warp lists the slice positions of
      // its keys in or above b* (in index order, in kbin, which the fast path does not
      // otherwise use) and counts the keys above b*; keys in b* also go to this CTA's
      // candidate list
      int ab = 0;
      // four rounds per iteration, their shared-memory loads issued together
      for (int j00 = w0; j00 < w1; j00 += 128) {
        unsigned kq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j = j00 + 32 * q + lane;
          kq[q] = j < w1 ? keys[j] : 0u;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j = j00 + 32 * q + lane;
          const unsigned key = kq[q], pre = key >> (32 - kPrefixBits);
          const bool isa = j < w1 && pre > bstar, isc = j < w1 && pre == bstar;
          const unsigned ba = __ballot_sync(0xffffffffu, isa), bs = ba | __ballot_sync(0xffffffffu, isc);
          if (isa || isc) kbin[w0 + nsel + __popc(bs & lt)] = (unsigned short)j;
          if (isc) {
            const int slot = atomicAdd(&sh_cand, 1);
            if (slot < kCandMax) cand[slot] = key;
          }
          nsel += __popc(bs);
          ab += __popc(ba);
        }
      }
      if (lane == 0) scan_buf[warp] = ab;
      __syncthreads();
      if (threadIdx.x == 0) {
        int sum = 0;
        for (int w = 0; w < nwarps; ++w) sum += scan_buf[w];
        sh_myab = sum;
      }
      cl.sync();   // S3: every CTA's list and count above b* are final
      // every CTA has read the row's prefix histogram: leave it zeroed for the next call
      for (int e = rank * (kPrefixBins / CS) + (int)threadIdx.x; e < (rank + 1) * (kPrefixBins / CS); e += blockDim.x)
        ghist[(long long)row * kPrefixBins + e] = 0u;
      if (threadIdx.x < 16) {
        const int r = (int)threadIdx.x;
        above_r[r] = r < CS ? *cl.map_shared_rank(&sh_cand, r) : 0;   // list lengths
        gt_r[r] = r < CS ? *cl.map_shared_rank(&sh_myab, r) : 0;      // keys above b*
      }
      __syncthreads();
      long long lsum = 0, asum = 0;
      for (int r = 0; r < CS; ++r) { lsum += above_r[r]; asum += gt_r[r]; }
      // the lists and counts come from the keys themselves: b* is the threshold bin iff
      // fewer than k keys lie above it and at least k lie in or above it (this holds
      // whatever the histogram held)
      ok = lsum == total && asum == sh_above && asum < k && asum + lsum >= k;   // the same in every CTA
      if (ok) {
        // every candidate is fetched by one thread (all remote loads in flight at once)
        static_assert(2 * kBins >= kCandMax && 4 * kBins >= kCandMax, "gather arrays fit in hist[1..3]");
        unsigned *allc = &hist[1][0];                                           // [kCandMax] gathered keys
        unsigned char *allr = reinterpret_cast<unsigned char *>(&hist[3][0]);   // ... and their ranks
        int offs[17];
        offs[0] = 0;
#pragma unroll
        for (int r = 0; r < 16; ++r) offs[r + 1] = offs[r] + above_r[r];
        for (int x = threadIdx.x; x < total; x += blockDim.x) {
          int r = 0;
#pragma unroll
          for (int q = 1; q < 16; ++q) r += x >= offs[q] ? 1 : 0;
          int base_r = 0;
#pragma unroll
          for (int q = 0; q < 16; ++q) base_r = q == r ? offs[q] : base_r;
          allc[x] = cl.map_shared_rank(cand, r)[x - base_r];
          allr[x] = (unsigned char)r;
        }
        cl.barrier_arrive();   // done reading peers' lists; the matching wait is at the very end
        fast_offsets = true;
        fast_list = true;
        __syncthreads();
        select_among(allc, allr, total, kin, bstar << (32 - kPrefixBits), ~0u << (32 - kPrefixBits));
      }
    } else {
      cl.sync();   // every CTA has read the row's prefix histogram
      for (int e = rank * (kPrefixBins / CS) + (int)threadIdx.x; e < (rank + 1) * (kPrefixBins / CS); e += blockDim.x)
        ghist[(long long)row * kPrefixBins + e] = 0u;
    }
    need_radix = !ok;
  } else {
    cl.sync();   // S1: every CTA's (min, max) visible; every part[] / counter zeroed
    if (ghist) {   // every CTA has read the row's prefix histogram: leave it zeroed for the next call
      for (int e = rank * (kPrefixBins / CS) + (int)threadIdx.x; e < (rank + 1) * (kPrefixBins / CS); e += blockDim.x)
        ghist[(long long)row * kPrefixBins + e] = 0u;
    }
    unsigned gmin = 0xFFFFFFFFu, gmax = 0u;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      if (r < CS) {
        const unsigned *mm = cl.map_shared_rank(sh_minmax, r);
        gmin = min(gmin, mm[0]);
        gmax = max(gmax, mm[1]);
      }
    }
    const float vmin = key_float(gmin), vmax = key_float(gmax);
    const float scale = (float)kBins / (vmax - vmin);
    const bool binned = gmax > gmin && isfinite(scale) && scale > 0.f && isfinite(vmin) && isfinite(vmax);
    need_radix = !binned;
    if (binned) {
      // ---- value histogram (bin(v) is monotone in v); non-empty bins are added
      //      straight into the owner CTA's merged array
      const int per = kBins / CS;
      unsigned *hsub = hist[warp & 3];
      for (int j = threadIdx.x; j < len; j += blockDim.x) {
        const int bin = min(kBins - 1, (int)((key_float(keys[j]) - vmin) * scale));
        kbin[j] = (unsigned short)bin;
        atomicAdd(&hsub[bin], 1u);
      }
      __syncthreads();
      for (int e = threadIdx.x; e < kBins; e += blockDim.x) {
        const unsigned v = hist[0][e] + hist[1][e] + hist[2][e] + hist[3][e];
        hist[0][e] = v;
        if (v) atomicAdd(cl.map_shared_rank(part, e / per) + e, v);
      }
      cl.sync();   // S2: merged histogram complete
      // thread x owns bins 2047-2x and 2046-2x (descending)
      const int b0 = kBins - 1 - 2 * (int)threadIdx.x, b1 = b0 - 1;
      const unsigned c0 = cl.map_shared_rank(part, b0 / per)[b0];
      const unsigned c1 = cl.map_shared_rank(part, b1 / per)[b1];
      int tot;
      const int above = block_exclusive_scan((int)(c0 + c1), scan_buf, tot);   // keys in higher bins
      if (above < k && above + (int)(c0 + c1) >= k) {
        const bool first = above + (int)c0 >= k;
        sh_bin = first ? b0 : b1;
        sh_above = first ? above : above + (int)c0;
        sh_incount = (int)(first ? c0 : c1);
      }
      __syncthreads();
      const int bstar = sh_bin, kin = k - sh_above, total = sh_incount;
      if (total <= kCandMax) {
        // ---- the threshold bin's keys of every CTA (with their rank) and every CTA's
        //      count of keys above the bin go to rank 0
        unsigned *cand0 = cl.map_shared_rank(cand, 0);
        unsigned char *crank0 = cl.map_shared_rank(cand_rank, 0);
        int *cnt0 = cl.map_shared_rank(&sh_cand, 0);
        for (int j = threadIdx.x; j < len; j += blockDim.x)
          if (kbin[j] == bstar) {
            const int slot = atomicAdd(cnt0, 1);
            cand0[slot] = keys[j];
            crank0[slot] = (unsigned char)rank;
          }
        {
          int ab = 0;   // keys of this slice in bins above b*
          for (int e = bstar + 1 + (int)threadIdx.x; e < kBins; e += blockDim.x) ab += (int)hist[0][e];
          ab = warp_sum_int(ab);
          if (lane == 0) scan_buf[warp] = ab;
          __syncthreads();
          if (threadIdx.x == 0) {
            int sum = 0;
            for (int w = 0; w < nwarps; ++w) sum += scan_buf[w];
            cl.map_shared_rank(above_r, 0)[rank] = sum;
          }
        }
        cl.sync();   // S3: rank 0 holds all `total` candidates and every CTA's count above
        constexpr int kSlots = kCandMax / kTopkThreads;
        unsigned mine[kSlots];
        unsigned char mrank[kSlots];
#pragma unroll
        for (int slot = 0; slot < kSlots; ++slot) {
          const int x = (int)threadIdx.x + slot * (int)blockDim.x;
          mine[slot] = x < total ? cand0[x] : 0u;
          mrank[slot] = x < total ? crank0[x] : (unsigned char)0;
        }
        int ab_r = 0;
        if (threadIdx.x < 16 && (int)threadIdx.x < CS) ab_r = cl.map_shared_rank(above_r, 0)[threadIdx.x];
        cl.barrier_arrive();   // done reading rank 0; the matching wait is at the very end
        fast_offsets = true;
        __syncthreads();
#pragma unroll
        for (int slot = 0; slot < kSlots; ++slot) {
          const int x = (int)threadIdx.x + slot * (int)blockDim.x;
          if (x < total) { cand[x] = mine[slot]; cand_rank[x] = mrank[slot]; }
        }
        if (threadIdx.x < 16) gt_r[threadIdx.x] = ab_r;
        __syncthreads();
        select_among(cand, cand_rank, total, kin, 0u, 0u);
      } else {
        need_radix = true;
      }
    }
  }
  if (need_radix) {
    // ---- fallback: three radix passes (11, 11, 10 bits) on the ordered keys
    unsigned mask = 0;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    const int per = kBins / CS;
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = shifts[pass];
      const unsigned dmask = (1u << widths[pass]) - 1u;
      for (int e = threadIdx.x; e < kBins; e += blockDim.x) hist[0][e] = 0;
      cl.sync();   // peers are done reading the previous histogram
      for (int j = threadIdx.x; j < len; j += blockDim.x) {
        const unsigned key = keys[j];
        const bool in = (key & mask) == prefix;
        const unsigned bin = (key >> shift) & dmask;
        const unsigned act = __ballot_sync(__activemask(), in);
        if (in) {
          const unsigned peers = __match_any_sync(act, bin);
          if ((threadIdx.x & 31) == (unsigned)(__ffs(peers) - 1)) atomicAdd(&hist[0][bin], __popc(peers));
        }
      }
      cl.sync();
      for (int e = threadIdx.x; e < per; e += blockDim.x) {
        unsigned v[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) v[r] = r < CS ? cl.map_shared_rank(&hist[0][0], r)[rank * per + e] : 0u;
        unsigned sum = 0;
#pragma unroll
        for (int r = 0; r < 16; ++r) sum += v[r];
        part[rank * per + e] = sum;
      }
      cl.sync();
      const int b0 = kBins - 1 - 2 * (int)threadIdx.x, b1 = b0 - 1;
      const unsigned c0 = cl.map_shared_rank(part, b0 / per)[b0];
      const unsigned c1 = cl.map_shared_rank(part, b1 / per)[b1];
      int tot;
      const int above = block_exclusive_scan((int)(c0 + c1), scan_buf, tot);
      if (above < krem && above + (int)(c0 + c1) >= krem) {
        const bool first = above + (int)c0 >= krem;
        sh_prefix = prefix | ((unsigned)(first ? b0 : b1) << shift);
        sh_krem = krem - (first ? above : above + (int)c0);
      }
      cl.sync();   // digit published; peers done reading part
      prefix = sh_prefix;
      krem = sh_krem;
      mask |= dmask << shift;
    }
  }
  // prefix = T, the k-th largest key; krem keys equal to T are still to be taken.
  // Each warp counts its keys > T and == T and compacts their slice positions, in
  // index order, to the front of its own run of keys[] (in place: a round writes
  // only below the keys it has still to read; bit 31 marks a key == T).  It walks
  // either its whole run or, on the fast path, only its list of keys in or above the
  // threshold bin.  One block scan orders the warps; the output pass walks the
  // compacted lists.
  int gw = 0, ew = 0;   // this warp's counts of keys > T and == T
  if (fast_list) {
    for (int i0 = 0; i0 < nsel; i0 += 32) {
      const int i = i0 + lane;
      const int j = i < nsel ? (int)kbin[w0 + i] : 0;
      const unsigned key = i < nsel ? keys[j] : 0u;
      const bool isg = i < nsel && key > prefix, ise = i < nsel && key == prefix;
      const unsigned bg = __ballot_sync(0xffffffffu, isg), be = __ballot_sync(0xffffffffu, ise);
      const unsigned bs = bg | be;
      if (isg || ise) keys[w0 + gw + ew + __popc(bs & lt)] = (unsigned)j | (ise ? 0x80000000u : 0u);
      gw += __popc(bg);
      ew += __popc(be);
    }
  } else {
    for (int j0 = w0; j0 < w1; j0 += 32) {
      const int j = j0 + lane;
      const unsigned key = j < w1 ? keys[j] : 0u;
      const bool isg = j < w1 && key > prefix, ise = j < w1 && key == prefix;
      const unsigned bg = __ballot_sync(0xffffffffu, isg), be = __ballot_sync(0xffffffffu, ise);
      const unsigned bs = bg | be;
      if (isg || ise) keys[w0 + gw + ew + __popc(bs & lt)] = (unsigned)j | (ise ? 0x80000000u : 0u);
      gw += __popc(bg);
      ew += __popc(be);
    }
  }
  int tot;
  const int ex = block_exclusive_scan(lane == 0 ? ((ew << 16) | gw) : 0, scan_buf, tot);   // counts < 2^16
  const int wex = __shfl_sync(0xffffffffu, ex, 0);
  int pg[16], pe[16];
  if (fast_offsets) {
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      pg[r] = r < rank ? gt_r[r] : 0;
      pe[r] = r < rank ? eq_r[r] : 0;
    }
  } else {
    if (threadIdx.x == 0) { cnt[0] = tot & 0xFFFF; cnt[1] = tot >> 16; }
    cl.sync();
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      pg[r] = r < rank ? cl.map_shared_rank(cnt, r)[0] : 0;
      pe[r] = r < rank ? cl.map_shared_rank(cnt, r)[1] : 0;
    }
    cl.barrier_arrive();
  }
  long long base = 0;
  int eq_before = 0;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    base += pg[r] + max(0, min(pe[r], krem - eq_before));
    eq_before += pe[r];
  }
  const int limit = max(0, krem - eq_before);   // equal keys this CTA may take, in index order
  int e_seen = wex >> 16;                        // equal keys before this warp's run (in this CTA)
  long long pos = base + (wex & 0xFFFF) + min(limit, e_seen);
  const int nw = gw + ew;                        // this warp's compacted list: keys[w0, w0 + nw)
  for (int i0 = 0; i0 < nw; i0 += 32) {
    const int i = i0 + lane;
    const unsigned ent = i < nw ? keys[w0 + i] : 0u;
    const bool ise = i < nw && (ent >> 31) != 0u, isg = i < nw && !ise;
    const unsigned be = __ballot_sync(0xffffffffu, ise);
    const bool take = isg || (ise && e_seen + __popc(be & lt) < limit);
    const unsigned bt = __ballot_sync(0xffffffffu, take);
    if (take) out[pos + __popc(bt & lt)] = (int32_t)(lo + (ent & 0x7FFFFFFFu));
    pos += __popc(bt);
    e_seen += __popc(be);
  }
  if (rank == 0 && threadIdx.x == 0) out_count[row] = k;
  cl.barrier_wait();   // no CTA leaves while a peer may still read its shared memory
}

// Row-split version (fused call, the indexer's prefix histograms at hand).  CTA p of a
// row takes its scores [p * kSplitChunk, (p + 1) * kSplitChunk), one per thread per
// slot, and no CTA waits for another:
//   1. the histogram gives the threshold bin b* (the prefix bin of the k-th largest
//      key); its loads, the scores' and the row length's are all in flight at once;
//   2. the CTA lists its keys in or above b*, in index order, as (index, key) entries
//      in its own block of the row's list, adds the next 11 bits of each key in b* to
//      the row's digit counts, and records its counts in its slot;
//   3. it takes a ticket; the row's last CTA (every other CTA's writes fenced before
//      their tickets) checks the counts against the histogram, reads the digit of the
//      k-th key from the digit counts and its last 8 bits from the listed keys of that
//      digit, which gives T, the k-th largest key; then it writes the list in order:
//      keys > T, then keys == T lowest index first.
// The counts come from the keys themselves, so a histogram that does not match them,
// or a bin with more than kCandMax keys, sends the last CTA to the single-CTA radix
// select over the whole row: a stale histogram costs time, never correctness.  Every
// decision is integer counting on the same data, whatever the order of arrival.
__global__ void __launch_bounds__(kTopkThreads) k_topk_split(CacheView c, int n_q, const float *scores,
                                                             long long stride, int k, int32_t *out_idx,
                                                             int32_t *out_count, TopkArea area, const int *status) {
  constexpr int kSlots = kSplitChunk / kTopkThreads;
  constexpr int kWarps = kTopkThreads / 32;
  constexpr int kRun = kSplitRun;
  static_assert(kSlots * kWarps <= kTopkThreads, "one thread per (slot, warp) count in the offset scan");
  static_assert(kPrefixBins == 8 * kTopkThreads && kDigitBins == 2 * kTopkThreads, "bins per thread");
  static_assert(kPrefixBits + 11 + 8 == 32, "prefix, digit and last bits make up a key");
  __shared__ int wcnt[kSlots * kWarps];          // entries per (slot, warp), then their offsets
  __shared__ int scan_buf[64];
  __shared__ int2 scan_buf2[64];
  __shared__ int sh_bin, sh_above, sh_incount;   // b*, keys above b*, keys in b* (histogram)
  __shared__ int sh_cnt[2];                      // this CTA's keys above b* and in b*
  __shared__ int sh_last;
  __shared__ int pos[kSplitPartsMax + 1];        // last CTA: each part's first position in the row's list
  __shared__ int lsum[3];                        // ... sums of the parts' counts; a part without a list
  __shared__ unsigned lhist[256];                // ... last 8 bits of the keys of the threshold digit
  __shared__ int sh_digit, sh_kr, sh_krem;
  __shared__ unsigned sh_T;
  const int p = blockIdx.x, row = blockIdx.y;
  const int b = row / n_q, i = row % n_q;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  pdl_wait();
  pdl_trigger();
  // ---- every load issued before any is needed: the row length, the status word, this
  //      thread's 8 histogram bins (descending over threads) and its scores (up to the
  //      row's capacity; keys past the row's length are masked below)
  unsigned *hrow = area.hist + (long long)row * kPrefixBins;
  const int hb = kPrefixBins - 8 * ((int)threadIdx.x + 1);
  const long long n_tok = c.n_tokens[b];
  const bool failed = status_failed(status);   // the same word for every CTA
  const uint4 h0 = *reinterpret_cast<const uint4 *>(hrow + hb);
  const uint4 h1 = *reinterpret_cast<const uint4 *>(hrow + hb + 4);
  const long long lo = (long long)p * kSplitChunk;
  const float *s = scores + (long long)row * stride + lo;
  const long long lim = min((long long)kSplitChunk, stride - lo);
  float v[kSlots];
#pragma unroll
  for (int q = 0; q < kSlots; ++q) {
    const int j = q * kTopkThreads + (int)threadIdx.x;
    v[q] = j < lim ? __ldg(s + j) : 0.f;
  }
  long long n = min((n_tok - n_q + i + 1) / c.m, c.cap);
  if (n > stride) n = stride;
  int32_t *out = out_idx + (long long)row * k;
  auto zero_hist = [&]() {   // leave the row's histogram zeroed for the next call
    for (int e = 4 * (int)threadIdx.x; e < kPrefixBins; e += 4 * kTopkThreads)
      *reinterpret_cast<uint4 *>(hrow + e) = make_uint4(0u, 0u, 0u, 0u);
  };
  if (n <= k || failed) {   // uniform over the row's CTAs; part 0 alone answers
    if (p == 0) {
      for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = (j < n && !failed) ? j : -1;
      if (threadIdx.x == 0) out_count[row] = failed ? -1 : (int32_t)n;
      zero_hist();   // the indexer counted this row's scores all the same
    }
    return;
  }
  const int parts = (int)((n + kSplitChunk - 1) / kSplitChunk);
  if (p >= parts) return;
  const int len = (int)min((long long)kSplitChunk, n - lo);
  // ---- 1. threshold bin from the histogram
  if (threadIdx.x == 0) { sh_bin = -1; sh_cnt[0] = 0; sh_cnt[1] = 0; }
  {
    const unsigned cb[8] = {h1.w, h1.z, h1.y, h1.x, h0.w, h0.z, h0.y, h0.x};   // descending bins
    int s8 = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) s8 += (int)cb[q];
    int tot;
    const int above = block_exclusive_scan(s8, scan_buf, tot);   // keys in higher bins
    if ((long long)tot == n && above < k && above + s8 >= k) {
      int cum = above;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (cum < k && cum + (int)cb[q] >= k) { sh_bin = hb + 7 - q; sh_above = cum; sh_incount = (int)cb[q]; }
        cum += (int)cb[q];
      }
    }
  }
  __syncthreads();
  const int bstar = sh_bin;                                   // -1: the histogram does not count n keys
  const bool hvalid = bstar >= 0 && sh_incount <= kCandMax;   // uniform
  int4 *slot = area.slots + (long long)row * area.parts + p;
  // ---- 2. this CTA's list: keys in or above b*, ordered by (slot, warp, lane) = index order
  if (hvalid) {
    unsigned key[kSlots], bsel[kSlots];
    int wa = 0, wi = 0;   // this warp's keys above b* and in b*
    unsigned *drow = area.dhist + (long long)row * kDigitBins;
#pragma unroll
    for (int q = 0; q < kSlots; ++q) {
      const int j = q * kTopkThreads + (int)threadIdx.x;
      key[q] = float_key(v[q]);
      const unsigned pre = key[q] >> (32 - kPrefixBits);
      const bool isin = j < len && pre == (unsigned)bstar;
      bsel[q] = __ballot_sync(0xffffffffu, j < len && pre >= (unsigned)bstar);
      const unsigned bin_ = __ballot_sync(0xffffffffu, isin);
      if (isin) atomicAdd(drow + ((key[q] >> 8) & (kDigitBins - 1)), 1u);
      if (lane == 0) wcnt[q * kWarps + warp] = __popc(bsel[q]);
      wa += __popc(bsel[q]) - __popc(bin_);
      wi += __popc(bin_);
    }
    if (lane == 0 && (wa | wi)) { atomicAdd(&sh_cnt[0], wa); atomicAdd(&sh_cnt[1], wi); }
    __syncthreads();
    const int vcnt = (int)threadIdx.x < kSlots * kWarps ? wcnt[threadIdx.x] : 0;
    int my_n;
    const int ex = block_exclusive_scan(vcnt, scan_buf, my_n);
    if ((int)threadIdx.x < kSlots * kWarps) wcnt[threadIdx.x] = ex;
    const bool room = my_n <= area.part_cap;   // uniform
    if (threadIdx.x == 0) *slot = make_int4(room ? my_n : -1, sh_cnt[0], sh_cnt[1], 0);
    __syncthreads();
    if (room) {
      uint2 *dst = area.lists + ((long long)row * area.parts + p) * area.part_cap;
#pragma unroll
      for (int q = 0; q < kSlots; ++q)
        if ((bsel[q] >> lane) & 1u)
          dst[wcnt[q * kWarps + warp] + __popc(bsel[q] & lt)] =
              make_uint2((unsigned)(lo + q * kTopkThreads + (int)threadIdx.x), key[q]);
    }
  } else if (threadIdx.x == 0) {
    *slot = make_int4(-1, 0, 0, 0);
  }
  // ---- 3. ticket (the grid-sync pattern: a CTA barrier, then one thread's fence and
  //      atomic); the row's last CTA resolves the row
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    sh_last = atomicAdd(&area.ctr[4 * row], 1u) == (unsigned)(parts - 1);
    if (sh_last) __threadfence();
  }
  __syncthreads();
  if (!sh_last) return;
  // ---- 4. the row's last CTA: the parts' counts and the digit counts
  if (threadIdx.x == 0) { lsum[0] = 0; lsum[1] = 0; lsum[2] = 0; sh_digit = -1; }
  if (threadIdx.x < 256) lhist[threadIdx.x] = 0u;
  int4 sl = make_int4(0, 0, 0, 0);
  if ((int)threadIdx.x < parts) sl = __ldcg(area.slots + (long long)row * area.parts + threadIdx.x);
  const unsigned *drow = area.dhist + (long long)row * kDigitBins;
  const int d0 = kDigitBins - 1 - 2 * (int)threadIdx.x, d1 = d0 - 1;   // this thread's digits, descending
  const int c0 = (int)__ldcg(drow + d0), c1 = (int)__ldcg(drow + d1);
  int2 tot2;
  const int2 ex2 = block_exclusive_scan2(make_int2(max(sl.x, 0), c0 + c1), scan_buf2, tot2);
  if ((int)threadIdx.x < parts) {
    pos[threadIdx.x] = ex2.x;
    atomicAdd(&lsum[0], sl.y);
    atomicAdd(&lsum[1], sl.z);
    if (sl.x < 0) lsum[2] = 1;
  }
  if (threadIdx.x == 0) pos[parts] = tot2.x;
  const int kin = k - sh_above;   // keys of b* to take
  if (hvalid && ex2.y < kin && ex2.y + c0 + c1 >= kin) {
    const bool first = ex2.y + c0 >= kin;
    sh_digit = first ? d0 : d1;
    sh_kr = kin - (first ? ex2.y : ex2.y + c0);
  }
  __syncthreads();
  // b* is the threshold bin iff fewer than k keys lie above it and at least k in or
  // above it; the parts' own counts decide, whatever the histogram held
  const bool ok = hvalid && lsum[2] == 0 && lsum[0] == sh_above && lsum[1] == sh_incount && sh_digit >= 0;
  if (!ok) {
    radix_select_row(scores + (long long)row * stride, n, k, out);
  } else {
    // this thread's contiguous run of the row's list (index order), held in registers
    const int N = tot2.x;   // < k + kCandMax <= kRun * kTopkThreads
    const int R = (N + kTopkThreads - 1) / kTopkThreads;
    const int x0 = min(N, (int)threadIdx.x * R), x1 = min(N, x0 + R);
    uint2 e[kRun];
#pragma unroll
    for (int r = 0; r < kRun; ++r) {
      const int x = x0 + r;
      e[r] = make_uint2(0u, 0u);
      if (x < x1) {
        int a0 = 0, a1 = parts - 1;   // the part holding x: the last with pos[q] <= x
        while (a0 < a1) {
          const int mid = (a0 + a1 + 1) >> 1;
          if (pos[mid] <= x) a0 = mid; else a1 = mid - 1;
        }
        e[r] = __ldcg(area.lists + ((long long)row * area.parts + a0) * area.part_cap + (x - pos[a0]));
      }
    }
    // the last 8 bits of the k-th key, from the listed keys of its digit
    const unsigned D = ((unsigned)bstar << 11) | (unsigned)sh_digit;
#pragma unroll
    for (int r = 0; r < kRun; ++r)
      if (x0 + r < x1 && (e[r].y >> 8) == D) atomicAdd(&lhist[e[r].y & 255u], 1u);
    __syncthreads();
    const int kr = sh_kr;
    const int cv = threadIdx.x < 256 ? (int)lhist[255 - threadIdx.x] : 0;
    int tot3;
    const int ab3 = block_exclusive_scan(cv, scan_buf, tot3);
    if (threadIdx.x < 256 && ab3 < kr && ab3 + cv >= kr) {
      sh_T = (D << 8) | (255u - threadIdx.x);
      sh_krem = kr - ab3;
    }
    __syncthreads();
    const unsigned T = sh_T;   // keys > T all go; krem keys == T go, lowest index first
    const int krem = sh_krem;
    int gt = 0, eq = 0;
#pragma unroll
    for (int r = 0; r < kRun; ++r)
      if (x0 + r < x1) { gt += e[r].y > T; eq += e[r].y == T; }
    int2 tot4;
    const int2 ex4 = block_exclusive_scan2(make_int2(gt, eq), scan_buf2, tot4);
    int po = ex4.x + min(ex4.y, krem), eq_seen = ex4.y;
#pragma unroll
    for (int r = 0; r < kRun; ++r) {
      if (x0 + r < x1) {
        if (e[r].y > T) {
          out[po++] = (int32_t)e[r].x;
        } else if (e[r].y == T) {
          if (eq_seen < krem) out[po++] = (int32_t)e[r].x;
          ++eq_seen;
        }
      }
    }
  }
  if (threadIdx.x == 0) out_count[row] = k;
  zero_hist();   // every CTA of the row read it before its ticket
}

namespace {
size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }
long long split_parts(int rows, long long n_cap, int k) {   // 0: no row-split area
  const long long parts = (n_cap + kSplitChunk - 1) / kSplitChunk;
  // the last CTA holds the row's list (< k + kCandMax entries) 8 entries per thread
  return rows >= 1 && parts >= 1 && parts <= kSplitPartsMax && k >= 1 && k + kCandMax <= kSplitRun * kTopkThreads
             ? parts
             : 0;
}
int part_cap(int k) { return k + kCandMax < kSplitChunk ? k + kCandMax : kSplitChunk; }
}  // namespace

size_t topk_area_bytes(int rows, long long n_cap, int k) {
  if (rows < 1 || rows > kPrefixRowsMax) return 0;
  size_t bytes = (size_t)rows * kPrefixBins * sizeof(unsigned);
  const long long parts = split_parts(rows, n_cap, k);
  if (parts)
    bytes += al256((size_t)rows * (4 + kDigitBins) * sizeof(unsigned)) + al256((size_t)rows * parts * sizeof(int4)) +
             (size_t)rows * parts * part_cap(k) * sizeof(uint2);
  return bytes;
}

TopkArea topk_area(void *base, int rows, long long n_cap, int k) {
  TopkArea a;
  a.rows = rows;
  a.hist = static_cast<unsigned *>(base);
  const long long parts = split_parts(rows, n_cap, k);
  if (parts) {
    char *q = static_cast<char *>(base) + (size_t)rows * kPrefixBins * sizeof(unsigned);
    a.ctr = reinterpret_cast<unsigned *>(q);
    a.dhist = a.ctr + (size_t)rows * 4;
    q += al256((size_t)rows * (4 + kDigitBins) * sizeof(unsigned));
    a.slots = reinterpret_cast<int4 *>(q);
    q += al256((size_t)rows * parts * sizeof(int4));
    a.lists = reinterpret_cast<uint2 *>(q);
    a.parts = (int)parts;
    a.part_cap = part_cap(k);
  }
  return a;
}

// With the indexer's prefix histograms and a row-split area (fused calls): the row-
// split kernel.  Otherwise rows with few queries get a cluster of up to 16 CTAs each;
// many rows get one CTA each.  Rows whose slice would not fit in shared memory use
// k_topk_row.
cudaError_t launch_topk(const CacheView &c, int batch, int n_q, const float *scores, long long stride, int k,
                        int32_t *out_idx, int32_t *out_count, const TopkArea *area, int num_sms, const int *status,
                        cudaStream_t st) {
  const int rows = batch * n_q;
  const long long n_cap = c.cap < stride ? c.cap : stride;
  unsigned *hist = area ? area->hist : nullptr;
  if (area && hist && area->parts > 0 && area->rows == rows && area->part_cap == part_cap(k) &&
      k + kCandMax <= kSplitRun * kTopkThreads && (long long)area->parts * kSplitChunk >= n_cap)
    return launch_pdl(k_topk_split, dim3(area->parts, rows), dim3(kTopkThreads), 0, st, 1, c, n_q, scores, stride, k,
                      out_idx, out_count, *area, status);
  // the row kernel does not read the indexer's prefix histograms; they are left zeroed
  // for the next call all the same
  auto row_kernel = [&]() -> cudaError_t {
    if (hist) {
      const cudaError_t e = cudaMemsetAsync(hist, 0, (size_t)rows * kPrefixBins * sizeof(unsigned), st);
      if (e != cudaSuccess) return e;
    }
    return launch_pdl(k_topk_row, dim3(rows), dim3(kRowThreads), 0, st, 1, c, n_q, scores, stride, k, out_idx,
                      out_count, status);
  };
  // cluster size: up to 16 CTAs per row for few rows; with many rows, halve it while
  // the grid exceeds two waves and the halved slices still fit in shared memory
  constexpr long long kSliceMax = 160 * 1024 / 6;   // uint32 key + uint16 bin per score
  int cs = 1;
  if (rows < num_sms) {
    cs = 16;
    while (cs > 1 && (long long)rows * cs > 2LL * num_sms && (n_cap + cs / 2 - 1) / (cs / 2) <= kSliceMax) cs /= 2;
  }
  const long long slice = (n_cap + cs - 1) / cs;
  const size_t smem = (size_t)slice * 6;   // uint32 key + uint16 bin per score
  if (smem > 160 * 1024 || cs > 16 || kBins % cs) return row_kernel();
  cudaError_t e = cudaFuncSetAttribute(k_topk_cluster, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
  if (e == cudaSuccess && cs > 8)
    e = cudaFuncSetAttribute(k_topk_cluster, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  for (;; cs /= 2) {
    const size_t sm = (size_t)((n_cap + cs - 1) / cs) * 6;
    if (sm > 160 * 1024) break;
    e = launch_pdl(k_topk_cluster, dim3(cs, rows), dim3(kTopkThreads), sm, st, cs, c, n_q, scores, stride, k, out_idx,
                   out_count, hist, (int)((n_cap + cs - 1) / cs), status);
    if (e == cudaSuccess || cs == 1) return e;
    cudaGetLastError();   // cluster too large for this device: halve it
  }
  return row_kernel();
}

}  // namespace csa
