// a2 — lightning-indexer scoring, CUDA-core version (any d_idx <= 128, fp32 or
// e4m3 keys).  Used for the fp32 cache format, for prefill rows and wherever the
// tensor-core kernel does not apply.
//
// Sources: "DeepSeek V4: How They Crushed the Million-Token Memory Problem"
// (sameershanbhag.com), "Two kinds of memory instead of one" — the lightning
// indexer scores compressed blocks with ReLU multi-head dot products and keeps
// the top-k; "DeepSeek V4 infrastructure" (volanea.com), "Compression only works
// if the attention path is engineered end to end" — sparse selection through the
// indexer.
//
// score_j = sum_h w_h * ReLU(q_h . key_j).  With e4m3 keys key_j = s_j * code_j
// and s_j > 0, so score_j = s_j * sum_h w_h * ReLU(q_h . code_j): the scale is
// applied once per entry.
//
// One thread scores one entry; the query's heads and weights sit in shared
// memory as fp32.  grid = (entry tiles, batch * n_q).
#include "kernels.h"

namespace csa {

template <int DI>
__global__ void __launch_bounds__(256) k_index_generic(CacheView c, int n_q, const uint8_t *q_idx, int q_dtype,
                                                       const float *w, int heads_idx, float *scores,
                                                       long long stride) {
  extern __shared__ float sm[];
  float *qs = sm;                            // [heads_idx][DI]
  float *ws = sm + heads_idx * DI;           // [heads_idx]
  const int row = blockIdx.y;                // b * n_q + i
  const int b = row / n_q, i = row % n_q;
  pdl_wait();
  pdl_trigger();
  const long long t = c.n_tokens[b] - n_q + i;
  const long long n_vis = min((t + 1) / c.m, c.cap);
  const long long j = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if ((long long)blockIdx.x * blockDim.x >= n_vis) return;   // whole CTA past the visible entries
  for (int e = threadIdx.x; e < heads_idx * DI; e += blockDim.x)
    qs[e] = load_tok(q_idx, q_dtype, (long long)row * heads_idx * DI + e);
  for (int e = threadIdx.x; e < heads_idx; e += blockDim.x) ws[e] = w[(long long)row * heads_idx + e];
  __syncthreads();
  if (q_dtype == CSA_BF16_Q_E4M3) {   // query-side FP8: each head's vector on the e4m3 grid of a power-of-two scale
    for (int h = threadIdx.x; h < heads_idx; h += blockDim.x) {
      float am = 0.f;
      for (int e = 0; e < DI; ++e) am = fmaxf(am, fabsf(qs[h * DI + e]));
      int ex = 0;
      frexpf(am, &ex);
      const float S = am > 0.f ? ldexpf(1.f, 8 - ex) : 1.f, inv = am > 0.f ? ldexpf(1.f, ex - 8) : 1.f;
      for (int e = 0; e < DI; ++e) qs[h * DI + e] = e4m3_to_f32(f32_to_e4m3_rn_sat(qs[h * DI + e] * S)) * inv;
    }
    __syncthreads();
  }
  if (j >= n_vis) return;
  const long long r = entry_row(c, b, j);
  float k[DI];
  float scale = 1.f;
  if (c.idx_fp4) {   // FP4 keys: DI/2 bytes, two e2m1 codes each
    const uint32_t *src = reinterpret_cast<const uint32_t *>(c.idx_key + r * (DI / 2));
#pragma unroll
    for (int v = 0; v < DI / 8; ++v) {
      const uint32_t wd = __ldg(src + v);
#pragma unroll
      for (int q = 0; q < 8; ++q) k[v * 8 + q] = e2m1_to_f32(wd >> (4 * q));
    }
    scale = __ldg(c.idx_scale + r);
  } else if (c.kv_dtype == CSA_E4M3) {
    const uint4 *src = reinterpret_cast<const uint4 *>(c.idx_key + r * DI);
#pragma unroll
    for (int v = 0; v < DI / 16; ++v) {
      const uint4 u = __ldg(src + v);
      const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int by = 0; by < 4; ++by) k[v * 16 + q * 4 + by] = e4m3_to_f32((wd[q] >> (8 * by)) & 0xFF);
    }
    scale = __ldg(c.idx_scale + r);
  } else {
    const float4 *src = reinterpret_cast<const float4 *>(c.idx_key) + r * (DI / 4);
#pragma unroll
    for (int v = 0; v < DI / 4; ++v) {
      const float4 f = __ldg(src + v);
      k[4 * v] = f.x; k[4 * v + 1] = f.y; k[4 * v + 2] = f.z; k[4 * v + 3] = f.w;
    }
  }
  float acc = 0.f;
  for (int h = 0; h < heads_idx; ++h) {
    const float *qh = qs + h * DI;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < DI; ++e) dot = fmaf(qh[e], k[e], dot);
    acc = fmaf(ws[h], fmaxf(dot, 0.f), acc);
  }
  scores[(long long)row * stride + j] = acc * scale;
}

cudaError_t launch_index_generic(const CacheView &c, int batch, int n_q, const void *q_idx, int q_dtype,
                                 const float *w, int heads_idx, float *scores, long long stride,
                                 long long n_cap, cudaStream_t st) {
  const int threads = 256;
  dim3 grid((unsigned)((n_cap + threads - 1) / threads), batch * n_q);
  const size_t smem = (size_t)heads_idx * (c.d_idx + 1) * sizeof(float);
  switch (c.d_idx) {
#define CASE(D)                                                                                              \
  case D:                                                                                                    \
    if (smem > 48 * 1024)                                                                                    \
      cudaFuncSetAttribute(k_index_generic<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);      \
    {                                                                                                        \
      cudaError_t e = launch_pdl(k_index_generic<D>, grid, dim3(threads), smem, st, 1, c, n_q,               \
                                 (const uint8_t *)q_idx, q_dtype, w, heads_idx, scores, stride);             \
      if (e != cudaSuccess) return e;                                                                        \
    }                                                                                                        \
    break;
    CASE(16) CASE(32) CASE(64) CASE(128)
#undef CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace csa
