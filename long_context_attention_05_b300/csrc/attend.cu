// a4 / a5 — shared-KV multi-query attention over compressed entries, the
// sliding window and the attention sink; CUDA-core (fp32) version.
//
// Sources: "DeepSeek V4 infrastructure" (volanea.com), "Compression only works
// if the attention path is engineered end to end" — shared key-value
// multi-query attention, partial rotary embeddings, sliding-window branch,
// attention sink; "DeepSeek V4: How They Crushed the Million-Token Memory
// Problem" (sameershanbhag.com), "Two kinds of memory instead of one" — CSA
// attends to the top-k blocks plus a window of uncompressed recent tokens; HCA
// attends densely to all 128-token entries with the same window.
//
// Key space of one query row: u < n_win are the window tokens t-n_win+1 .. t,
// n_win <= u < n_win + n_list the entries (CSA: idx[row][u - n_win], HCA: entry
// u - n_win), the order the tensor-core kernel uses.  A CTA
// handles HG heads of one row and a contiguous range of KC-key chunks with an
// online softmax; with one split it also adds the sink and writes the output,
// otherwise it writes (max, sum, weighted sum) partials that k_attend_combine
// merges in fixed split order (deterministic).
#include "kernels.h"

namespace csa {

constexpr int kAttThreads = 256;

__global__ void __launch_bounds__(kAttThreads) k_attend(AttendArgs a) {
  extern __shared__ float sm[];
  const CacheView &c = a.c;
  const int d = c.d, dr = c.d_rope, dn = d - dr, ks_ld = d + 1;
  float *qs = sm;                          // [kHG][d]
  float *ks = qs + kHG * d;                // [kKC][d+1]
  float *ps = ks + kKC * ks_ld;            // [kHG][kKC]
  float *m_run = ps + kHG * kKC;           // [kHG]
  float *l_run = m_run + kHG;              // [kHG]
  float *corr = l_run + kHG;               // [kHG]
  long long *ksrc = reinterpret_cast<long long *>(corr + kHG);   // [kKC] row (>=0), -2-pos (window), -1 none

  const int row = blockIdx.z;
  const int b = row / a.n_q, iq = row % a.n_q;
  pdl_wait();
  pdl_trigger();
  const long long t = c.n_tokens[b] - a.n_q + iq;
  const long long n_vis = min((t + 1) / c.m, c.cap);
  const long long n_list = a.idx ? a.k : n_vis;
  const long long U = n_list + c.n_win;
  const int h0 = blockIdx.y * kHG;
  const int nh = min(kHG, a.heads - h0);
  const int split = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // splits past this row's keys (the plan covers the key-list capacity) do nothing;
  // the merge reads only the splits that hold keys
  if (a.idx == nullptr && a.n_splits > 1 && (long long)split * a.keys_per_split >= U) return;   // uniform (dense rows)

  // query heads, rotated at t
  for (int e = tid; e < nh * d; e += blockDim.x)
    qs[e] = load_tok(a.q, a.q_dtype, ((long long)row * a.heads + h0) * d + e);
  if (tid < kHG) { m_run[tid] = -INFINITY; l_run[tid] = 0.f; }
  __syncthreads();
  for (int p = tid; p < nh * (dr / 2); p += blockDim.x) {
    const int hh = p / (dr / 2), pr = p % (dr / 2);
    float cs, sn;
    rope_cos_sin(t, a.rope.step[pr], cs, sn);
    float *v = qs + hh * d + dn + 2 * pr;
    const float x0 = v[0], x1 = v[1];
    v[0] = fmaf(x0, cs, -x1 * sn);
    v[1] = fmaf(x0, sn, x1 * cs);
  }
  constexpr int R = 4;   // d <= 1024 = R * 256
  float acc[kHG][R];
#pragma unroll
  for (int hh = 0; hh < kHG; ++hh)
#pragma unroll
    for (int r = 0; r < R; ++r) acc[hh][r] = 0.f;

  const long long ch0 = (long long)split * a.chunks_per_split;
  for (long long chunk = ch0; chunk < ch0 + a.chunks_per_split; ++chunk) {
    const long long u0 = chunk * kKC;
    if (u0 >= U) break;
    __syncthreads();
    if (tid < kKC) {
      const long long u = u0 + tid;
      long long src = -1;
      if (u < c.n_win) {
        const long long tau = t - c.n_win + 1 + u;
        if (tau >= 0) src = -2 - tau;
      } else if (u < U) {
        const long long e = u - c.n_win;
        const long long j = a.idx ? (long long)a.idx[(long long)row * a.k + e] : e;
        if (j >= 0 && j < n_vis) src = entry_row(c, b, j);
      }
      ksrc[tid] = src;
    }
    __syncthreads();
    for (int x = tid; x < kKC * d; x += blockDim.x) {
      const int kk = x / d, e = x % d;
      const long long src = ksrc[kk];
      float v = 0.f;
      if (src >= 0) {
        if (c.kv_dtype == CSA_E4M3)
          v = e < dn ? e4m3_to_f32(__ldg(c.kv_nope + src * dn + e)) * __ldg(c.kv_scale + src)
                     : bf16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t *>(c.kv_rope) + src * dr + (e - dn)));
        else
          v = e < dn ? __ldg(reinterpret_cast<const float *>(c.kv_nope) + src * dn + e)
                     : __ldg(reinterpret_cast<const float *>(c.kv_rope) + src * dr + (e - dn));
      } else if (src <= -2) {
        const long long tau = -2 - src;
        v = load_tok(c.win, c.win_dtype, ((long long)b * c.win_cap + tau % c.win_cap) * d + e);
      }
      ks[kk * ks_ld + e] = v;
    }
    __syncthreads();
    for (int p = tid; p < kKC * (dr / 2); p += blockDim.x) {   // window keys turn at their own position
      const int kk = p / (dr / 2), pr = p % (dr / 2);
      const long long src = ksrc[kk];
      if (src <= -2) {
        float cs, sn;
        rope_cos_sin(-2 - src, a.rope.step[pr], cs, sn);
        float *v = ks + kk * ks_ld + dn + 2 * pr;
        const float x0 = v[0], x1 = v[1];
        v[0] = fmaf(x0, cs, -x1 * sn);
        v[1] = fmaf(x0, sn, x1 * cs);
      }
    }
    __syncthreads();
    // logits: warp w handles heads w and w+8, lane = key
    for (int hh = warp; hh < nh; hh += kAttThreads / 32) {
      const float *qh = qs + hh * d;
      const float *kr = ks + lane * ks_ld;
      float dot = 0.f;
      for (int e = 0; e < d; ++e) dot = fmaf(qh[e], kr[e], dot);
      const bool valid = ksrc[lane] != -1;
      const float sl = valid ? dot * a.scale : -INFINITY;
      const float cmax = warp_max(sl);
      const float m_old = m_run[hh];
      const float m_new = fmaxf(m_old, cmax);
      const float p = (valid && m_new > -INFINITY) ? expf(sl - m_new) : 0.f;
      const float cr = (m_old > -INFINITY) ? expf(m_old - m_new) : (m_new > -INFINITY ? 0.f : 1.f);
      const float psum = warp_sum(p);
      ps[hh * kKC + lane] = p;
      if (lane == 0) { corr[hh] = cr; l_run[hh] = l_run[hh] * cr + psum; m_run[hh] = m_new; }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int e = tid + r * kAttThreads;
      if (e < d) {
#pragma unroll
        for (int hh = 0; hh < kHG; ++hh) {
          if (hh < nh) {
            float s = acc[hh][r] * corr[hh];
#pragma unroll 8
            for (int kk = 0; kk < kKC; ++kk) s = fmaf(ps[hh * kKC + kk], ks[kk * ks_ld + e], s);
            acc[hh][r] = s;
          }
        }
      }
    }
  }
  __syncthreads();
  if (a.n_splits == 1) {
#pragma unroll
    for (int hh = 0; hh < kHG; ++hh) {
      if (hh >= nh) break;
      const int h = h0 + hh;
      const float z = __ldg(a.sink + h);
      const float M = fmaxf(m_run[hh], z);
      const float L = l_run[hh] * (m_run[hh] > -INFINITY ? expf(m_run[hh] - M) : 0.f) + expf(z - M);
      const float f = (m_run[hh] > -INFINITY ? expf(m_run[hh] - M) : 0.f) / L;
      const long long ob = ((long long)row * a.heads + h) * d;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int e = tid + r * kAttThreads;
        if (e < d) {
          const float o = acc[hh][r] * f;
          if (a.out_dtype == CSA_F32) reinterpret_cast<float *>(a.out)[ob + e] = o;
          else reinterpret_cast<uint16_t *>(a.out)[ob + e] = f32_to_bf16_rn(o);
        }
      }
      if (tid == 0 && a.out_lse) a.out_lse[(long long)row * a.heads + h] = M + logf(L);
    }
  } else {
#pragma unroll
    for (int hh = 0; hh < kHG; ++hh) {
      if (hh >= nh) break;
      const int h = h0 + hh;
      const long long pb = ((long long)row * a.n_splits + split) * a.heads + h;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int e = tid + r * kAttThreads;
        if (e < d) a.part_o[pb * d + e] = acc[hh][r];
      }
      if (tid == 0) { a.part_ml[pb * 2] = m_run[hh]; a.part_ml[pb * 2 + 1] = l_run[hh]; }
    }
  }
}

// Merge of split partials: M = max(sink, m_s), L = exp(sink-M) + sum_s l_s exp(m_s-M),
// out = sum_s o_s exp(m_s-M) / L, lse = M + log L.  One CTA of 512 threads per
// (row, pair of heads) -- one wave on the GPU for a decode batch -- and a thread
// owns two adjacent output elements of one head, with up to 16 partial loads (8
// bytes each) in flight: the merge costs a few memory round trips, not one per
// split.  Every sum has a fixed shape (per element: s = 0, 1, ... in order; L:
// per-thread strided sums, then a fixed tree), so the bits do not depend on
// timing or on the batch.
constexpr int kCombThreads = 512;
constexpr int kCombHeads = 2;   // heads per CTA
__global__ void __launch_bounds__(kCombThreads) k_attend_combine(AttendArgs a) {
  extern __shared__ float wts[];   // [kCombHeads][n_splits] (the first S of each used)
  __shared__ float red[kCombHeads][2][kCombThreads / 32];
  const int row = blockIdx.y;
  const int d = a.c.d;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = kCombThreads / 32;
  // thread layout: head slot hs = tid / (kCombThreads / kCombHeads); element pair e2 within the head
  constexpr int TPH = kCombThreads / kCombHeads;
  const int hs = tid / TPH, t2 = tid % TPH;
  const int h = blockIdx.x * kCombHeads + hs;
  const bool hv = h < a.heads;
  const int SP = a.n_splits;   // stride of the partial arrays
  const long long base = (long long)row * SP * a.heads + h;
  // this thread's first split's (m, l) and the sink load together with n_tokens
  const float z = hv ? __ldg(a.sink + h) : 0.f;
  const float2 ml0 = hv && t2 < SP ? *reinterpret_cast<const float2 *>(a.part_ml + (base + (long long)t2 * a.heads) * 2)
                                  : make_float2(-INFINITY, 0.f);
  // only the splits that hold keys of this row were written (the same count the
  // attention kernel derives from n_tokens)
  const int bq = row / a.n_q, iq = row % a.n_q;
  const long long t = a.c.n_tokens[bq] - a.n_q + iq;
  const long long U = (a.idx ? a.k : min((t + 1) / a.c.m, a.c.cap)) + a.c.n_win;
  const int S = (int)max(0LL, min((long long)SP, (U + a.keys_per_split - 1) / a.keys_per_split));
  // this thread's first element pair of the first kPre splits' partial outputs, issued
  // before the weights that scale them are known (every partial of a split below S is
  // written and finite, so a zero weight takes it out exactly)
  constexpr int kPre = 32;
  float2 pre[kPre];
  const bool pre_ok = hv && 2 * t2 < d;
#pragma unroll
  for (int q = 0; q < kPre; ++q)
    pre[q] = pre_ok && q < S ? *reinterpret_cast<const float2 *>(a.part_o + (base + (long long)q * a.heads) * d + 2 * t2)
                             : make_float2(0.f, 0.f);
  // per head: M and the split weights (the threads of a head are whole warps)
  float m = z;
  if (hv) {
    if (t2 < S) m = fmaxf(m, ml0.x);
    for (int s = t2 + TPH; s < S; s += TPH) m = fmaxf(m, a.part_ml[(base + (long long)s * a.heads) * 2]);
  }
  m = warp_max(m);
  if (lane == 0) red[hs][0][warp % (NW / kCombHeads)] = m;
  __syncthreads();
  float M = red[hs][0][0];
#pragma unroll
  for (int i = 1; i < NW / kCombHeads; ++i) M = fmaxf(M, red[hs][0][i]);
  float lp = 0.f;
  if (hv) {
    for (int s = t2; s < S; s += TPH) {
      const float2 ml = s == t2 ? ml0 : *reinterpret_cast<const float2 *>(a.part_ml + (base + (long long)s * a.heads) * 2);
      const float ws = ml.x > -INFINITY ? expf(ml.x - M) : 0.f;
      wts[hs * S + s] = ws;
      lp = fmaf(ws, ml.y, lp);
    }
  }
  lp = warp_sum(lp);
  if (lane == 0) red[hs][1][warp % (NW / kCombHeads)] = lp;
  __syncthreads();
  float L = expf(z - M);
#pragma unroll
  for (int i = 0; i < NW / kCombHeads; ++i) L += red[hs][1][i];
  const float invL = 1.f / L;
  const float *w = wts + hs * S;
  for (int e = 2 * t2; hv && e < d; e += 2 * TPH) {
    float o0 = 0.f, o1 = 0.f;
    int s_from = 0;
    if (e == 2 * t2) {   // the preloaded splits, in split order
#pragma unroll
      for (int q = 0; q < kPre; ++q)
        if (q < S) {
          o0 = fmaf(w[q], pre[q].x, o0);
          o1 = fmaf(w[q], pre[q].y, o1);
        }
      s_from = kPre;
    }
    for (int s0 = s_from; s0 < S; s0 += 16) {
      float2 v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q)
        v[q] = (s0 + q < S && w[s0 + q] != 0.f)
                   ? *reinterpret_cast<const float2 *>(a.part_o + (base + (long long)(s0 + q) * a.heads) * d + e)
                   : make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (s0 + q < S) {
          o0 = fmaf(w[s0 + q], v[q].x, o0);
          o1 = fmaf(w[s0 + q], v[q].y, o1);
        }
    }
    o0 *= invL;
    o1 *= invL;
    const long long ob = ((long long)row * a.heads + h) * d + e;
    if (a.out_dtype == CSA_F32) *reinterpret_cast<float2 *>(reinterpret_cast<float *>(a.out) + ob) = make_float2(o0, o1);
    else *reinterpret_cast<uint32_t *>(reinterpret_cast<uint16_t *>(a.out) + ob) =
             (uint32_t)f32_to_bf16_rn(o0) | ((uint32_t)f32_to_bf16_rn(o1) << 16);
  }
  if (hv && t2 == 0 && a.out_lse) a.out_lse[(long long)row * a.heads + h] = M + logf(L);
}

// Split plan shared by the launcher and the workspace sizing.  It depends only
// on the key-list capacity, on whether the call is a decode (one query per
// sequence) and on `wide` (a dense call -- every visible entry, no top-k list --
// with d >= 256), never on the batch, so a row's reduction order -- and its bits
// -- do not change with the other rows in the batch.  Decode: two 64-key chunks
// per CTA (tensor-core kernel; four for wide calls, whose long key lists would
// otherwise write d-wide partials for every 128 keys) or four 32-key chunks
// (CUDA-core kernel), merged by k_attend_combine.  Prefill (many queries per sequence): one CTA walks all
// chunks of its row.  The window comes first in a row's key list, so splits past
// the last key hold only absent keys: a longer list of the same keys adds splits
// whose partials weigh exactly zero in the merge.
void attend_plan(int n_q, long long list_cap, int n_win, bool tc, bool wide, int &n_splits, int &cps) {
  const int keys = tc ? 64 : kKC;               // keys per chunk of the kernel that runs
  const long long chunks = (list_cap + n_win + keys - 1) / keys;
  if (n_q > 1) {
    cps = (int)chunks;
    n_splits = 1;
    return;
  }
  cps = tc ? (wide ? 4 : 2) : 4;
  n_splits = (int)((chunks + cps - 1) / cps);
}

size_t attend_smem_bytes(int d) {
  return ((size_t)kHG * d + (size_t)kKC * (d + 1) + kHG * kKC + 3 * kHG) * sizeof(float) + kKC * sizeof(long long);
}

cudaError_t launch_attend(const AttendArgs &a0, int rows, cudaStream_t st) {
  AttendArgs a = a0;
  const size_t smem = attend_smem_bytes(a.c.d);
  cudaFuncSetAttribute(k_attend, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 grid(a.n_splits, (a.heads + kHG - 1) / kHG, rows);
  cudaError_t e = launch_pdl(k_attend, grid, dim3(kAttThreads), smem, st, 1, a);
  if (e != cudaSuccess || a.n_splits == 1) return e;
  return launch_attend_combine(a, rows, st);
}

cudaError_t launch_attend_combine(const AttendArgs &a, int rows, cudaStream_t st) {
  return launch_pdl(k_attend_combine, dim3((a.heads + kCombHeads - 1) / kCombHeads, rows), dim3(kCombThreads),
                    kCombHeads * a.n_splits * sizeof(float), st, 1, a);
}

}  // namespace csa
