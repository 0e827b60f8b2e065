// a1 — softmax-gated block pooling fused into the KV-cache append.
//
// Sources: "DeepSeek Releases V4 with Million-Token Context Optimized for AI
// Agents" (botbeat.news), Summary — CSA compresses 4 tokens into one entry by
// softmax-gated pooling with a learned positional bias; "DeepSeek V4: How They
// Crushed the Million-Token Memory Problem" (sameershanbhag.com), "Two kinds of
// memory instead of one" — 4 (CSA) / 128 (HCA) tokens per entry, fp8 KV with
// bf16 rotary dims; "DeepSeek V4 infrastructure" (volanea.com), "Compression
// only works if the attention path is engineered end to end" — partial RoPE and
// state caches for the sliding window.
//
// One CTA owns one block (m tokens) of one sequence; thread c owns channel c of
// the KV stream (c < d) or of the indexer-key stream (d <= c < d + d_idx).  The
// pooling runs as an online softmax (running max, sum and weighted sum per
// channel) so a block can be fed one token per decode step; the running state
// of the block in progress lives in cache->pool_state between calls.
//
// CTA 0 of each sequence owns both the first block the call touches (which may
// continue from pool_state) and the last one (which may leave a partial block
// in pool_state), so pool_state is read and written by a single CTA.  With one
// new token there is one CTA per sequence, and it advances n_tokens itself;
// otherwise a one-thread-per-sequence kernel advances it after the pooling.
#include "kernels.h"

namespace csa {

struct CompressArgs {
  CacheView c;
  RopeTable rope;
  int n_new;
  int in_dtype;
  const uint8_t *x, *gate, *idx_x, *idx_gate;
  const float *pos_bias, *idx_pos_bias;
};

__device__ __forceinline__ float block_max(float v, float *red) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float r = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r = fmaxf(r, red[i]);
  return r;
}

// Pools (the rest of) block j for this thread's channel and, when the block is
// complete, writes the entry.  Called by all threads of the CTA (uniform j).
__device__ void pool_block(const CompressArgs &a, int b, long long n0, long long j, bool from_state,
                           bool write_state, float *xs, float *red) {
  const CacheView &c = a.c;
  const int ch = threadIdx.x;
  const int dch = c.d + c.d_idx;
  const bool active = ch < dch;
  const bool kv = ch < c.d;
  const long long p_lo = max(j * c.m, n0), p_hi = min((j + 1) * c.m, n0 + a.n_new);
  const bool complete = (j + 1) * c.m <= n0 + a.n_new;
  float mx = 0.f, sum = 0.f, acc = 0.f;
  float *st = c.pool_state + (long long)b * 3 * dch;
  if (active && from_state) {
    mx = st[ch];
    sum = st[dch + ch];
    acc = st[2 * dch + ch];
  }
  if (active) {
    const long long ring_lo = n0 + a.n_new - c.win_cap;
    for (long long p = p_lo; p < p_hi; ++p) {
      const long long i = p - n0;   // token index within this call
      float xv, lg;
      if (kv) {
        const long long off = ((long long)b * a.n_new + i) * c.d + ch;
        xv = load_tok(a.x, a.in_dtype, off);
        lg = load_tok(a.gate, a.in_dtype, off) + __ldg(a.pos_bias + (p - j * c.m));
        if (p >= ring_lo) {   // raw token into the window ring (same dtype as the input)
          const long long slot = ((long long)b * c.win_cap + p % c.win_cap) * c.d + ch;
          if (a.in_dtype == CSA_F32)
            reinterpret_cast<float *>(const_cast<uint8_t *>(c.win))[slot] = xv;
          else
            reinterpret_cast<uint16_t *>(const_cast<uint8_t *>(c.win))[slot] =
                __ldg(reinterpret_cast<const uint16_t *>(a.x) + off);
        }
      } else {
        const long long off = ((long long)b * a.n_new + i) * c.d_idx + (ch - c.d);
        xv = load_tok(a.idx_x, a.in_dtype, off);
        lg = load_tok(a.idx_gate, a.in_dtype, off) + __ldg(a.idx_pos_bias + (p - j * c.m));
      }
      if (sum == 0.f) {
        mx = lg; sum = 1.f; acc = xv;
      } else if (lg > mx) {
        const float r = expf(mx - lg);
        acc = acc * r + xv; sum = sum * r + 1.f; mx = lg;
      } else {
        const float e = expf(lg - mx);
        acc = fmaf(e, xv, acc); sum += e;
      }
    }
  }
  if (!complete) {
    if (active && write_state) { st[ch] = mx; st[dch + ch] = sum; st[2 * dch + ch] = acc; }
    return;
  }
  // finished entry: value, rotary turn of the last d_rope KV dims at position j*m
  float e = active ? acc / sum : 0.f;
  const int rope0 = c.d - c.d_rope;
  if (active) xs[ch] = e;
  __syncthreads();
  if (kv && ch >= rope0) {
    const int pr = (ch - rope0) >> 1;
    const float a0 = xs[rope0 + 2 * pr], a1 = xs[rope0 + 2 * pr + 1];
    float cs, sn;
    rope_cos_sin(j * c.m, a.rope.step[pr], cs, sn);
    e = ((ch - rope0) & 1) ? fmaf(a0, sn, a1 * cs) : fmaf(a0, cs, -a1 * sn);
  }
  if (j >= c.cap) return;   // no room: entry dropped (capacity is the caller's contract)
  const long long row = entry_row(c, b, j);
  if (c.kv_dtype == CSA_E4M3) {
    const float amax_kv = block_max((kv && ch < rope0) ? fabsf(e) : 0.f, red);
    const float amax_ix = block_max((active && !kv) ? fabsf(e) : 0.f, red);
    float s_kv = amax_kv / 448.0f, s_ix = amax_ix / (c.idx_fp4 ? 6.0f : 448.0f);
    if (!(s_kv >= 1.17549435e-38f)) s_kv = 1.0f;
    if (!(s_ix >= 1.17549435e-38f)) s_ix = 1.0f;
    if (kv && ch < rope0) {
      const_cast<uint8_t *>(c.kv_nope)[row * rope0 + ch] = f32_to_e4m3_rn_sat(e / s_kv);
      if (ch == 0) const_cast<float *>(c.kv_scale)[row] = s_kv;
    } else if (kv) {
      reinterpret_cast<uint16_t *>(const_cast<uint8_t *>(c.kv_rope))[row * c.d_rope + (ch - rope0)] =
          f32_to_bf16_rn(e);
    } else if (active && !c.idx_fp4) {
      const_cast<uint8_t *>(c.idx_key)[row * c.d_idx + (ch - c.d)] = f32_to_e4m3_rn_sat(e / s_ix);
      if (ch == c.d) const_cast<float *>(c.idx_scale)[row] = s_ix;
    }
    if (c.idx_fp4) {   // two e2m1 codes per byte: the even channel writes its own and its neighbour's
      const uint32_t code = (active && !kv) ? f32_to_e2m1_rn_sat(e / s_ix) : 0u;
      const uint32_t next = __shfl_down_sync(0xffffffffu, code, 1);   // every lane takes part
      const int k = ch - c.d;
      if (active && !kv && (k & 1) == 0)
        const_cast<uint8_t *>(c.idx_key)[row * (c.d_idx / 2) + k / 2] = (uint8_t)(code | (next << 4));
      if (ch == c.d) const_cast<float *>(c.idx_scale)[row] = s_ix;
    }
  } else {
    if (kv && ch < rope0)
      reinterpret_cast<float *>(const_cast<uint8_t *>(c.kv_nope))[row * rope0 + ch] = e;
    else if (kv)
      reinterpret_cast<float *>(const_cast<uint8_t *>(c.kv_rope))[row * c.d_rope + (ch - rope0)] = e;
    else if (active)
      reinterpret_cast<float *>(const_cast<uint8_t *>(c.idx_key))[row * c.d_idx + (ch - c.d)] = e;
  }
  if (write_state && active) { st[ch] = 0.f; st[dch + ch] = 0.f; st[2 * dch + ch] = 0.f; }
}

__global__ void __launch_bounds__(1024) k_compress(CompressArgs a) {
  extern __shared__ float smem[];
  float *xs = smem;                 // [d + d_idx]
  float *red = smem + 1024;         // [32]
  const int b = blockIdx.y;
  pdl_wait();      // the previous step's attention reads the ring and n_tokens
  pdl_trigger();
  const long long n0 = a.c.n_tokens[b];
  const long long j0 = n0 / a.c.m, j1 = (n0 + a.n_new - 1) / a.c.m;
  if (blockIdx.x == 0) {
    pool_block(a, b, n0, j0, j0 * a.c.m < n0, j1 == j0, xs, red);
    if (j1 != j0) {
      __syncthreads();
      pool_block(a, b, n0, j1, false, true, xs, red);
    }
    if (gridDim.x == 1) {   // single new token: this CTA is the only reader of n_tokens[b]
      __syncthreads();
      if (threadIdx.x == 0) a.c.n_tokens[b] = n0 + a.n_new;
    }
  } else {
    const long long j = j0 + blockIdx.x;
    if (j < j1) pool_block(a, b, n0, j, false, false, xs, red);
  }
}

// Sliding-window-only layer: the raw tokens go into the window ring (the last win_cap
// of them) and n_tokens advances; nothing is pooled.  One CTA per sequence reads
// n_tokens first and advances it after every copy of the sequence is issued.
__global__ void __launch_bounds__(256) k_swa_append(CacheView c, int n_new, int in_dtype, const uint8_t *x) {
  const int b = blockIdx.x;
  pdl_wait();      // the previous step's attention reads the ring and n_tokens
  pdl_trigger();
  __shared__ long long sh_n0;
  if (threadIdx.x == 0) sh_n0 = c.n_tokens[b];
  __syncthreads();
  const long long n0 = sh_n0;
  const long long first = max(0LL, (long long)n_new - c.win_cap);   // earlier tokens would be overwritten
  const int esz = in_dtype == CSA_F32 ? 4 : 2;
  const long long row_bytes = (long long)c.d * esz;                 // a multiple of 16 (d % 16 == 0)
  const long long n_vec = (n_new - first) * (row_bytes / 16);
  uint8_t *ring = const_cast<uint8_t *>(c.win);
  for (long long v = threadIdx.x; v < n_vec; v += blockDim.x) {
    const long long i = first + v / (row_bytes / 16), piece = v % (row_bytes / 16);
    const long long p = n0 + i;
    const uint4 val = __ldg(reinterpret_cast<const uint4 *>(x + ((long long)b * n_new + i) * row_bytes) + piece);
    reinterpret_cast<uint4 *>(ring + ((long long)b * c.win_cap + p % c.win_cap) * row_bytes)[piece] = val;
  }
  __syncthreads();
  if (threadIdx.x == 0) c.n_tokens[b] = n0 + n_new;
}

__global__ void k_advance(long long *n_tokens, int batch, int n_new) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch) n_tokens[b] += n_new;
}

cudaError_t launch_compress(const CacheView &c, const RopeTable &rope, int batch, int n_new, int in_dtype,
                            const void *x, const void *gate, const void *ix, const void *ig,
                            const float *pb, const float *ipb, cudaStream_t st) {
  CompressArgs a;
  a.c = c; a.rope = rope; a.n_new = n_new; a.in_dtype = in_dtype;
  a.x = (const uint8_t *)x; a.gate = (const uint8_t *)gate;
  a.idx_x = (const uint8_t *)ix; a.idx_gate = (const uint8_t *)ig;
  a.pos_bias = pb; a.idx_pos_bias = ipb;
  const int threads = ((c.d + c.d_idx + 31) / 32) * 32;
  const int nblk = n_new == 1 ? 1 : (n_new + c.m - 1) / c.m + 1;
  const size_t smem = (1024 + 32) * sizeof(float);
  cudaError_t e = launch_pdl(k_compress, dim3(nblk, batch), dim3(threads), smem, st, 1, a);
  if (e != cudaSuccess || n_new == 1) return e;
  k_advance<<<(batch + 127) / 128, 128, 0, st>>>(c.n_tokens, batch, n_new);
  return cudaGetLastError();
}

cudaError_t launch_swa_append(const CacheView &c, int batch, int n_new, int in_dtype, const void *x, cudaStream_t st) {
  return launch_pdl(k_swa_append, dim3(batch), dim3(256), 0, st, 1, c, n_new, in_dtype, (const uint8_t *)x);
}

}  // namespace csa
