// a4 / a5 — shared-KV multi-query attention on tensor cores (mma.sync f16).
//
// Sources: "DeepSeek V4 infrastructure" (volanea.com), "Compression only works
// if the attention path is engineered end to end" — shared key-value
// multi-query attention, partial RoPE, sliding-window branch, attention sink;
// "DeepSeek V4: How They Crushed the Million-Token Memory Problem"
// (sameershanbhag.com), "Two kinds of memory instead of one" — attention over
// the selected (CSA) or all (HCA) compressed entries plus the window.
//
// Work split.  A CTA = one query row x one group of 16 heads (one m16 tile) x one
// split of the row's key list (decode: two 64-key chunks; prefill: all chunks of
// the row).  Key list of a row: the window tokens first (oldest to newest), then
// the selected entries in list order (CSA) or all visible entries (HCA), so a key
// list padded with absent (-1) entries at the end leaves every chunk -- and every
// bit of the row's result -- unchanged.
//
// Operands are f16 with power-of-two scale factors, so no bf16 or e4m3-with-scale
// input overflows or underflows f16:
//   q            rotated at t in fp32, times S_h (max|q| S_h < 2^14)
//   entry nope   e4m3 code * 2^-8 (exact),           sigma_n = 2^8 * s_j (s_j its scale)
//   entry rope   bf16 value * 2^-e (per entry),       sigma_r = 2^e
//   window token raw bf16 nope dims * 2^-e_n, rotary dims turned at the token's
//                position then * 2^-e_r (per token), sigma_n = 2^e_n, sigma_r = 2^e_r
// (e chosen so the key's largest magnitude lands in [2^14, 2^15)).  Logits
//   l = (sigma_n S_nope + sigma_r S_rope) / (S_h sqrt(d))
// with the e4m3 and rotary parts accumulated separately.  Values are the same key
// rows (shared KV): the e4m3 dims take P * sigma_n, the rotary dims P * sigma_r,
// each divided by a per-(head, chunk) power of two 2^F that puts its largest
// product just below 1 before it is rounded to f16; the fp32 accumulators carry
// 2^F (rescaled with the online-softmax correction between chunks).
//
// 8 warps.  Logits: warp w computes the 16 heads x keys 8w..8w+7 of a chunk;
// softmax: 16 threads per head; values: warp w accumulates the 16 heads x dims
// w*d/8 .. (w+1)*d/8 in registers.  One split: the CTA adds the sink and writes
// the output; several: it writes (m, l, o) partials for k_attend_combine.
#include <climits>

#include "kernels.h"

namespace csa {
namespace {

constexpr int kTcHeads = 16;              // heads per CTA
constexpr int kKeys = 64;            // keys per chunk
constexpr int kThreads = 256;
constexpr int kTPK = kThreads / kKeys;   // gather threads per key
constexpr int kPadH = 8;             // f16 row padding (16 bytes) against bank conflicts
constexpr int kNoExp = -100000;      // "no exponent yet" of the value accumulators

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void ldm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// 2^e as a float, for |e| <= 126
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }

// Exponent e of a key's scale factor: its largest magnitude m times 2^-e lies in
// [2^14, 2^15) (clamped to |e| <= 100; 0 when m == 0).
__device__ __forceinline__ int key_exp(float m) {
  if (!(m > 0.f)) return 0;
  int e;
  frexpf(m, &e);   // m in [2^(e-1), 2^e)
  return max(-100, min(100, e - 15));
}

__device__ __forceinline__ float max4(float a, float b, float c, float d) { return fmaxf(fmaxf(a, b), fmaxf(c, d)); }

// max over the kTPK = 4 consecutive lanes that gather one key
__device__ __forceinline__ float key_group_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2) k_attend_tc(AttendArgs a) {
  constexpr int DN = D - 64;                 // e4m3 dims (rotary dims: the last 64)
  constexpr int LDQ = D + kPadH;             // f16 row stride of the Q and K tiles
  constexpr int LDP = kKeys + kPadH;         // f16 row stride of the P tiles
  constexpr int LDS = kKeys + 4;             // fp32 row stride of the logit tile
  constexpr int DW = D / 8;                  // dims per warp in the value phase
  constexpr int NT = DW / 8;                 // n-tiles per warp in the value phase
  constexpr int NOPE16 = DN / 16;            // 16-byte e4m3 pieces of an entry
  constexpr int NP_E = (NOPE16 + kTPK - 1) / kTPK;
  constexpr int NP_R = 8 / kTPK;             // 16-byte bf16 pieces of the rotary dims, per thread
  constexpr int NP_W = D / 8 / kTPK;         // 16-byte bf16 pieces of a window token, per thread
  constexpr int NBUF = NP_E + NP_R > NP_W ? NP_E + NP_R : NP_W;
  constexpr int QPER = D / 16;               // query dims per thread (16 threads per head)
  static_assert(DN % 32 == 0, "a window token's rotary pieces fall on whole threads");
  static_assert(NT % 2 == 0, "value n-tiles in pairs");

  extern __shared__ __align__(16) uint8_t smem[];
  // the rotary phase steps, read by every thread with its own pair index: from shared
  // memory (a lane-varying index into the kernel parameters serialises its loads)
  __shared__ unsigned long long rstep[32];
  __half *Qs = reinterpret_cast<__half *>(smem);                       // [16][LDQ]
  __half *Ks = Qs + kTcHeads * LDQ;                                          // [64][LDQ]
  float *Sf = reinterpret_cast<float *>(Ks + kKeys * LDQ);             // [16][LDS]
  __half *Pn = reinterpret_cast<__half *>(Sf + kTcHeads * LDS);             // [16][LDP] P sigma_n / 2^Fn
  __half *Pr = Pn + kTcHeads * LDP;                                          // [16][LDP] P sigma_r / 2^Fr
  float *sig_n = reinterpret_cast<float *>(Pr + kTcHeads * LDP);            // [64]
  float *sig_r = sig_n + kKeys;                                         // [64]
  float *qsc = sig_r + kKeys;                                           // [16] 1/(S_h sqrt d)
  float *m_run = qsc + kTcHeads;
  float *l_run = m_run + kTcHeads;
  float *c_n = l_run + kTcHeads;                                             // [16] correction, e4m3 dims
  float *c_r = c_n + kTcHeads;                                               // [16] correction, rotary dims
  int *f_n = reinterpret_cast<int *>(c_r + kTcHeads);                        // [16] exponent of the e4m3-dim accumulator
  int *f_r = f_n + kTcHeads;                                                 // [16] ... of the rotary-dim accumulator
  long long *ksrc = reinterpret_cast<long long *>(f_r + kTcHeads);          // [64]
  float2 *qcs = reinterpret_cast<float2 *>(ksrc + kKeys);              // [32] (cos, sin) at t
  float2 *wcs = qcs + 32;                                               // [64][32] window tokens' (cos, sin)

  const CacheView &c = a.c;
  const int row = blockIdx.x;              // rows in x: prefill calls can have more than 65535
  const int h0 = blockIdx.y * kTcHeads;
  const int b = row / a.n_q, iq = row % a.n_q;
  const int H = a.heads;
  const int split = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int W = c.n_win;

  // ---- the query rows of this head group: issued before anything else
  const int qh = tid >> 4, qpart = tid & 15;   // 16 threads per head, QPER dims each
  uint4 qraw[QPER / 8];
  const bool q_live = h0 + qh < H;
  if (a.q_dtype == CSA_BF16) {
#pragma unroll
    for (int u = 0; u < QPER / 8; ++u)
      qraw[u] = q_live ? __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(a.q) +
                                                               ((long long)row * H + h0 + qh) * D + qpart * QPER) + u)
                       : make_uint4(0, 0, 0, 0);
  }
  pdl_wait();
  pdl_trigger();
  const long long t = c.n_tokens[b] - a.n_q + iq;
  const long long n_vis = min((t + 1) / c.m, c.cap);
  const long long n_list = a.idx ? a.k : n_vis;
  const long long U = W + n_list;
  // splits past this row's keys (the plan covers the key-list capacity) do nothing;
  // the merge reads only the splits that hold keys.  Only a dense (HCA) row can end early.
  if (a.idx == nullptr && a.n_splits > 1 && (long long)split * a.keys_per_split >= U) return;   // uniform

  // key source of slot u of the row's key list: entry row (>= 0), -2 - ring row
  // (window token at position t - W + 1 + u), -1 (absent)
  auto key_src = [&](long long u, float &sn) {
    long long src = -1;
    sn = 0.f;
    if (u < W) {
      const long long tau = t - W + 1 + u;
      if (tau >= 0) src = -2 - ((long long)b * c.win_cap + tau % c.win_cap);
    } else if (u < U) {
      const long long e = u - W;
      const long long j = a.idx ? (long long)__ldg(a.idx + (long long)row * a.k + e) : e;
      if (j >= 0 && j < n_vis) {
        src = entry_row(c, b, j);
        sn = 256.f * __ldg(c.kv_scale + src);
      }
    }
    return src;
  };

  // ---- key gather: kTPK threads per key.  gather_load issues every load of this
  //      thread into registers; gather_store scales, converts and stores them.
  const int gk = tid / kTPK, gsub = tid % kTPK;
  auto gather_load = [&](uint4 (&buf)[NBUF]) {
    const long long src = ksrc[gk];
#pragma unroll
    for (int i = 0; i < NBUF; ++i) buf[i] = make_uint4(0, 0, 0, 0);
    if (src >= 0) {
#pragma unroll
      for (int i = 0; i < NP_E; ++i) {
        const int p = gsub + kTPK * i;
        if (p < NOPE16) buf[i] = __ldg(reinterpret_cast<const uint4 *>(c.kv_nope + src * DN) + p);
      }
#pragma unroll
      for (int r = 0; r < NP_R; ++r)
        buf[NP_E + r] = __ldg(reinterpret_cast<const uint4 *>(c.kv_rope + src * 64 * 2) + gsub + kTPK * r);
    } else if (src <= -2) {
#pragma unroll
      for (int i = 0; i < NP_W; ++i)
        buf[i] = __ldg(reinterpret_cast<const uint4 *>(c.win + (-2 - src) * D * 2) + gsub + kTPK * i);
    }
  };
  auto bf2f = [](uint32_t w, float &lo, float &hi) {
    lo = bf16_bits_to_f32((uint16_t)(w & 0xFFFF));
    hi = bf16_bits_to_f32((uint16_t)(w >> 16));
  };
  auto gather_store = [&](const uint4 (&buf)[NBUF]) {
    const long long src = ksrc[gk];
    __half *dst = Ks + gk * LDQ;
    const bool is_e = src >= 0, is_w = src <= -2;
    // rotary dims as fp32: an entry's stored (already turned) values, or a window
    // token's raw values turned at its position
    float rf[NP_R][8];
#pragma unroll
    for (int r = 0; r < NP_R; ++r) {
      const uint4 u = is_e ? buf[NP_E + r] : buf[NP_W - NP_R + r];
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) bf2f(w4[e], rf[r][2 * e], rf[r][2 * e + 1]);
      if (is_w) {
        const int pr0 = (gsub + kTPK * r) * 4;   // first rotary pair of this piece
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const float2 cs = wcs[gk * 32 + pr0 + e / 2];
          const float x0 = rf[r][e], x1 = rf[r][e + 1];
          rf[r][e] = fmaf(x0, cs.x, -x1 * cs.y);
          rf[r][e + 1] = fmaf(x0, cs.y, x1 * cs.x);
        }
      }
    }
    float mr = 0.f;
#pragma unroll
    for (int r = 0; r < NP_R; ++r)
#pragma unroll
      for (int e = 0; e < 8; ++e) mr = fmaxf(mr, fabsf(rf[r][e]));
    // window tokens: the largest magnitude of the non-rotary dims as well
    float mn = 0.f;
    if (is_w) {
#pragma unroll
      for (int i = 0; i < NP_W - NP_R; ++i) {
        const uint4 u = buf[i];
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float lo, hi;
          bf2f(w4[e], lo, hi);
          mn = fmaxf(mn, fmaxf(fabsf(lo), fabsf(hi)));
        }
      }
    }
    mr = key_group_max(mr);   // every lane takes part (keys of a warp differ in kind)
    mn = key_group_max(mn);
    const int er = key_exp(mr), en = key_exp(mn);
    const float inv_r = pow2i(-er), inv_n = pow2i(-en);
    if (is_e) {
#pragma unroll
      for (int i = 0; i < NP_E; ++i) {
        const int p = gsub + kTPK * i;
        if (p < NOPE16) {
          const uint4 u = buf[i];
          uint4 o0, o1;
          o0.x = e4m3x2_to_f16x2_scaled(u.x); o0.y = e4m3x2_to_f16x2_scaled(u.x >> 16);
          o0.z = e4m3x2_to_f16x2_scaled(u.y); o0.w = e4m3x2_to_f16x2_scaled(u.y >> 16);
          o1.x = e4m3x2_to_f16x2_scaled(u.z); o1.y = e4m3x2_to_f16x2_scaled(u.z >> 16);
          o1.z = e4m3x2_to_f16x2_scaled(u.w); o1.w = e4m3x2_to_f16x2_scaled(u.w >> 16);
          *reinterpret_cast<uint4 *>(dst + p * 16) = o0;
          *reinterpret_cast<uint4 *>(dst + p * 16 + 8) = o1;
        }
      }
    } else if (is_w) {
#pragma unroll
      for (int i = 0; i < NP_W - NP_R; ++i) {
        const uint4 u = buf[i];
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
        uint4 o;
        uint32_t *op = &o.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float lo, hi;
          bf2f(w4[e], lo, hi);
          op[e] = pack_h2(lo * inv_n, hi * inv_n);
        }
        *reinterpret_cast<uint4 *>(dst + (gsub + kTPK * i) * 8) = o;
      }
    } else {   // absent key: a zero row (its logits are masked; zeros keep P V finite)
#pragma unroll
      for (int i = 0; i < NP_W; ++i)
        *reinterpret_cast<uint4 *>(dst + (gsub + kTPK * i) * 8) = make_uint4(0, 0, 0, 0);
    }
    if (is_e || is_w) {
#pragma unroll
      for (int r = 0; r < NP_R; ++r) {
        uint4 o;
        o.x = pack_h2(rf[r][0] * inv_r, rf[r][1] * inv_r); o.y = pack_h2(rf[r][2] * inv_r, rf[r][3] * inv_r);
        o.z = pack_h2(rf[r][4] * inv_r, rf[r][5] * inv_r); o.w = pack_h2(rf[r][6] * inv_r, rf[r][7] * inv_r);
        *reinterpret_cast<uint4 *>(dst + DN + (gsub + kTPK * r) * 8) = o;
      }
    }
    if (gsub == 0) {
      if (is_w) sig_n[gk] = pow2i(en);   // entries: 2^8 s_j, set with the key lookup
      sig_r[gk] = (is_e || is_w) ? pow2i(er) : 0.f;
    }
  };
  // (cos, sin) of every rotary pair of the chunk's window tokens (slot u of the key
  // list sits at position t - W + 1 + u).  Thread x takes pair x % 32 of keys
  // x / 32 + KS r: the first angle is evaluated, the others follow by turning it KS
  // positions at a time (angle addition; relative error ~1e-6, far below the f16
  // rounding of the key operand).
  auto win_rope = [&](long long u0) {
    constexpr int KS = kThreads / 32;
    const int kk0 = tid >> 5, pr = tid & 31;
    float c0, s0, cd, sd;
    rope_cos_sin(t - W + 1 + u0 + kk0, rstep[pr], c0, s0);
    rope_cos_sin(KS, rstep[pr], cd, sd);
#pragma unroll
    for (int r = 0; r < kKeys / KS; ++r) {
      const int kk = kk0 + KS * r;
      if (ksrc[kk] <= -2) wcs[kk * 32 + pr] = make_float2(c0, s0);
      const float c1 = fmaf(c0, cd, -s0 * sd);
      s0 = fmaf(s0, cd, c0 * sd);
      c0 = c1;
    }
  };

  const long long ch0 = (long long)split * a.chunks_per_split;
  // ---- prologue: the first chunk's key lookups, the query's rotary table
  long long src_next = -1;
  float sn_next = 0.f;
  if (tid < kKeys) {
    float sn;
    const long long src = key_src(ch0 * kKeys + tid, sn);
    ksrc[tid] = src;
    sig_n[tid] = sn;
    if (a.chunks_per_split > 1) src_next = key_src((ch0 + 1) * kKeys + tid, sn_next);
  } else if (tid < kKeys + 32) {
    float cs, sn;
    rstep[tid - kKeys] = a.rope.step[tid - kKeys];
    rope_cos_sin(t, a.rope.step[tid - kKeys], cs, sn);
    qcs[tid - kKeys] = make_float2(cs, sn);
  }
  if (tid < kTcHeads) {
    m_run[tid] = -INFINITY;
    l_run[tid] = 0.f;
    f_n[tid] = kNoExp;
    f_r[tid] = kNoExp;
  }
  __syncthreads();   // ksrc, qcs, rstep
  uint4 gbuf[NBUF];
  gather_load(gbuf);
  const bool win0 = ch0 * kKeys < W;   // uniform: window tokens in the first chunk
  if (win0) win_rope(ch0 * kKeys);
  {   // ---- query: rotate, scale by a power of two per head, convert to f16
    float v[QPER];
    if (a.q_dtype == CSA_BF16) {
#pragma unroll
      for (int u = 0; u < QPER / 8; ++u) {
        const uint32_t w4[4] = {qraw[u].x, qraw[u].y, qraw[u].z, qraw[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) bf2f(w4[e], v[u * 8 + 2 * e], v[u * 8 + 2 * e + 1]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < QPER; ++e)
        v[e] = q_live ? __ldg(reinterpret_cast<const float *>(a.q) + ((long long)row * H + h0 + qh) * D + qpart * QPER + e)
                      : 0.f;
    }
    if (qpart * QPER + QPER > DN) {
#pragma unroll
      for (int e = 0; e < QPER; e += 2) {
        const int dim = qpart * QPER + e;
        if (dim >= DN) {
          const float2 cs = qcs[(dim - DN) >> 1];
          const float x0 = v[e], x1 = v[e + 1];
          v[e] = fmaf(x0, cs.x, -x1 * cs.y);
          v[e + 1] = fmaf(x0, cs.y, x1 * cs.x);
        }
      }
    }
    float am = 0.f;
#pragma unroll
    for (int e = 0; e < QPER; ++e) am = fmaxf(am, fabsf(v[e]));
#pragma unroll
    for (int o = 8; o; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    int ex = 0;
    frexpf(am, &ex);
    const float S = am > 0.f ? ldexpf(1.f, 14 - ex) : 1.f;   // max|q| S < 2^14
    uint32_t pk[QPER / 2];
#pragma unroll
    for (int e = 0; e < QPER; e += 2) pk[e / 2] = pack_h2(v[e] * S, v[e + 1] * S);
    uint4 *qd = reinterpret_cast<uint4 *>(Qs + qh * LDQ + qpart * QPER);
#pragma unroll
    for (int u = 0; u < QPER / 8; ++u) qd[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
    if (qpart == 0) qsc[qh] = a.scale / S;
  }
  if (win0) __syncthreads();   // window (cos, sin) table
  gather_store(gbuf);

  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[n][r] = 0.f;

  for (long long chunk = ch0; chunk < ch0 + a.chunks_per_split; ++chunk) {
    const long long u0 = chunk * kKeys;
    if (u0 >= U) break;
    __syncthreads();   // previous chunk's value phase done with Ks / P (first chunk: its tile stored)
    if (chunk != ch0) {
      if (tid < kKeys) {
        ksrc[tid] = src_next;
        sig_n[tid] = sn_next;
        src_next = -1;
        if (chunk + 1 < ch0 + a.chunks_per_split) src_next = key_src(u0 + kKeys + tid, sn_next);
      }
      __syncthreads();
      gather_load(gbuf);
      if (u0 < W) {   // uniform
        win_rope(u0);
        __syncthreads();
      }
      gather_store(gbuf);
      __syncthreads();
    }
    // ---- logits: warp w = heads 0..15 x keys 8w..8w+7; e4m3 part in two chains, rotary part in one
    {
      float an0[4] = {0.f, 0.f, 0.f, 0.f}, an1[4] = {0.f, 0.f, 0.f, 0.f}, ar[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t qa = su32(Qs + (lane & 15) * LDQ + (lane >> 4) * 8);
      const uint32_t kb = su32(Ks + (8 * warp + (lane & 7)) * LDQ + ((lane >> 3) & 1) * 8);
#pragma unroll 4
      for (int ks = 0; ks < DN / 16; ks += 2) {
        uint32_t a0, a1, a2, a3, b0, b1, c0, c1, c2, c3, d0, d1;
        ldm_x4(qa + ks * 32, a0, a1, a2, a3);
        ldm_x2(kb + ks * 32, b0, b1);
        ldm_x4(qa + ks * 32 + 32, c0, c1, c2, c3);
        ldm_x2(kb + ks * 32 + 32, d0, d1);
        mma16816(an0, a0, a1, a2, a3, b0, b1);
        mma16816(an1, c0, c1, c2, c3, d0, d1);
      }
#pragma unroll
      for (int ks = DN / 16; ks < D / 16; ++ks) {
        uint32_t a0, a1, a2, a3, b0, b1;
        ldm_x4(qa + ks * 32, a0, a1, a2, a3);
        ldm_x2(kb + ks * 32, b0, b1);
        mma16816(ar, a0, a1, a2, a3, b0, b1);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int h = (lane >> 2) + (r >= 2 ? 8 : 0);
        const int kk = 8 * warp + 2 * (lane & 3) + (r & 1);
        Sf[h * LDS + kk] = ksrc[kk] != -1 ? (sig_n[kk] * (an0[r] + an1[r]) + sig_r[kk] * ar[r]) * qsc[h] : -INFINITY;
      }
    }
    __syncthreads();
    // ---- online softmax: 16 threads per head, 4 keys each; P sigma scaled per head
    {
      const int h = tid >> 4, part = tid & 15;
      const float4 sv = *reinterpret_cast<const float4 *>(Sf + h * LDS + part * 4);
      const float l4[4] = {sv.x, sv.y, sv.z, sv.w};
      float cmax = max4(l4[0], l4[1], l4[2], l4[3]);
#pragma unroll
      for (int o = 8; o; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
      const float m_old = m_run[h];
      const float m_new = fmaxf(m_old, cmax);
      float p4[4], psum = 0.f, gn = 0.f, gr = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        p4[e] = (m_new > -INFINITY && l4[e] > -INFINITY) ? __expf(l4[e] - m_new) : 0.f;
        psum += p4[e];
        gn = fmaxf(gn, p4[e] * sig_n[part * 4 + e]);
        gr = fmaxf(gr, p4[e] * sig_r[part * 4 + e]);
      }
#pragma unroll
      for (int o = 8; o; o >>= 1) {
        psum += __shfl_xor_sync(0xffffffffu, psum, o);
        gn = fmaxf(gn, __shfl_xor_sync(0xffffffffu, gn, o));
        gr = fmaxf(gr, __shfl_xor_sync(0xffffffffu, gr, o));
      }
      // exponents F of this chunk's largest products (never more than 60 below the
      // accumulator's previous one, so the rescaling factor stays in range)
      const int fn_old = f_n[h], fr_old = f_r[h];
      int en, er;
      frexpf(gn, &en);
      frexpf(gr, &er);
      const int fn_new = gn > 0.f ? (fn_old == kNoExp ? en : max(en, fn_old - 60)) : fn_old;
      const int fr_new = gr > 0.f ? (fr_old == kNoExp ? er : max(er, fr_old - 60)) : fr_old;
      const float sn_inv = fn_new == kNoExp ? 0.f : ldexpf(1.f, -fn_new);
      const float sr_inv = fr_new == kNoExp ? 0.f : ldexpf(1.f, -fr_new);
      uint32_t pn[2], pr[2];
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        pn[e / 2] = pack_h2(p4[e] * sig_n[part * 4 + e] * sn_inv, p4[e + 1] * sig_n[part * 4 + e + 1] * sn_inv);
        pr[e / 2] = pack_h2(p4[e] * sig_r[part * 4 + e] * sr_inv, p4[e + 1] * sig_r[part * 4 + e + 1] * sr_inv);
      }
      *reinterpret_cast<uint2 *>(Pn + h * LDP + part * 4) = make_uint2(pn[0], pn[1]);
      *reinterpret_cast<uint2 *>(Pr + h * LDP + part * 4) = make_uint2(pr[0], pr[1]);
      __syncwarp();
      if (part == 0) {
        const float corr = m_old > -INFINITY ? __expf(m_old - m_new) : 0.f;
        c_n[h] = fn_old == kNoExp ? 0.f : ldexpf(corr, fn_old - fn_new);
        c_r[h] = fr_old == kNoExp ? 0.f : ldexpf(corr, fr_old - fr_new);
        l_run[h] = (m_old > -INFINITY ? l_run[h] * corr : 0.f) + psum;
        m_run[h] = m_new;
        f_n[h] = fn_new;
        f_r[h] = fr_new;
      }
    }
    __syncthreads();
    // ---- values: warp w = heads 0..15 x dims w*DW .. w*DW + DW - 1
    {
      const float cl_n = c_n[lane >> 2], ch_n = c_n[(lane >> 2) + 8];
      const float cl_r = c_r[lane >> 2], ch_r = c_r[(lane >> 2) + 8];
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const bool nope = warp * DW + n * 8 < DN;
        const float cl = nope ? cl_n : cl_r, chh = nope ? ch_n : ch_r;
        acc[n][0] *= cl; acc[n][1] *= cl;
        acc[n][2] *= chh; acc[n][3] *= chh;
      }
      const uint32_t pa_off = ((lane & 15) * LDP + (lane >> 4) * 8) * 2;
      const uint32_t pna = su32(Pn) + pa_off, pra = su32(Pr) + pa_off;
#pragma unroll
      for (int ks = 0; ks < kKeys / 16; ++ks) {
        uint32_t n0, n1, n2, n3, r0, r1, r2, r3;
        ldm_x4(pna + ks * 32, n0, n1, n2, n3);
        ldm_x4(pra + ks * 32, r0, r1, r2, r3);
        const uint32_t vb = su32(Ks + (ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LDQ + warp * DW + (lane >> 4) * 8);
#pragma unroll
        for (int n = 0; n < NT; n += 2) {
          uint32_t b0, b1, b2, b3;
          ldm_x4_t(vb + n * 16, b0, b1, b2, b3);
          const bool nope0 = warp * DW + n * 8 < DN, nope1 = warp * DW + (n + 1) * 8 < DN;
          if (nope0) mma16816(acc[n], n0, n1, n2, n3, b0, b1);
          else mma16816(acc[n], r0, r1, r2, r3, b0, b1);
          if (nope1) mma16816(acc[n + 1], n0, n1, n2, n3, b2, b3);
          else mma16816(acc[n + 1], r0, r1, r2, r3, b2, b3);
        }
      }
    }
  }
  __syncthreads();
  // ---- output (one split) or partials, in real units: accumulator * 2^F
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int hl = (lane >> 2) + 8 * half;
    const int h = h0 + hl;
    if (h >= H) continue;
    const float un = f_n[hl] == kNoExp ? 0.f : ldexpf(1.f, f_n[hl]);
    const float ur = f_r[hl] == kNoExp ? 0.f : ldexpf(1.f, f_r[hl]);
    float f = 1.f, lse = 0.f;
    if (a.n_splits == 1) {
      const float z = __ldg(a.sink + h);
      const float mr = m_run[hl];
      const float M = fmaxf(mr, z);
      const float em = mr > -INFINITY ? expf(mr - M) : 0.f;
      const float L = l_run[hl] * em + expf(z - M);
      f = em / L;
      lse = M + logf(L);
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int dim = warp * DW + n * 8 + 2 * (lane & 3);
      const float u = dim < DN ? un : ur;
      const float o0 = acc[n][2 * half] * u * f, o1 = acc[n][2 * half + 1] * u * f;
      if (a.n_splits == 1) {
        const long long ob = ((long long)row * H + h) * D + dim;
        if (a.out_dtype == CSA_F32) *reinterpret_cast<float2 *>(reinterpret_cast<float *>(a.out) + ob) = make_float2(o0, o1);
        else *reinterpret_cast<uint32_t *>(reinterpret_cast<uint16_t *>(a.out) + ob) =
                 (uint32_t)f32_to_bf16_rn(o0) | ((uint32_t)f32_to_bf16_rn(o1) << 16);
      } else {
        const long long pb = ((long long)row * a.n_splits + split) * H + h;
        *reinterpret_cast<float2 *>(a.part_o + pb * D + dim) = make_float2(o0, o1);
      }
    }
    if ((lane & 3) == 0 && warp == 0) {
      if (a.n_splits == 1) {
        if (a.out_lse) a.out_lse[(long long)row * H + h] = lse;
      } else {
        const long long pb = ((long long)row * a.n_splits + split) * H + h;
        a.part_ml[pb * 2] = m_run[hl];
        a.part_ml[pb * 2 + 1] = l_run[hl];
      }
    }
  }
}

}  // namespace

bool attend_tc_supported(const CacheView &c, int heads, int q_dtype) {
  return c.kv_dtype == CSA_E4M3 && c.win_dtype == CSA_BF16 && c.d_rope == 64 &&
         (c.d == 128 || c.d == 256 || c.d == 384 || c.d == 512) && heads >= 1 && heads <= 128 &&
         (q_dtype == CSA_BF16 || q_dtype == CSA_F32);
}

size_t attend_tc_smem_bytes(int d) {
  return (size_t)(kTcHeads + kKeys) * (d + kPadH) * 2 + (size_t)kTcHeads * (kKeys + 4) * 4 + (size_t)2 * kTcHeads * (kKeys + kPadH) * 2 +
         (size_t)2 * kKeys * 4 + (size_t)7 * kTcHeads * 4 + (size_t)kKeys * 8 + 32 * 8 + (size_t)kKeys * 32 * 8;
}

cudaError_t launch_attend_tc(const AttendArgs &a, int rows, cudaStream_t st) {
  const size_t smem = attend_tc_smem_bytes(a.c.d);
  if (a.n_splits > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid(rows, (a.heads + kTcHeads - 1) / kTcHeads, a.n_splits);
  cudaError_t e = cudaSuccess;
  switch (a.c.d) {
#define CASE(D)                                                                                   \
  case D:                                                                                         \
    e = cudaFuncSetAttribute(k_attend_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
    if (e != cudaSuccess) return e;                                                               \
    e = launch_pdl(k_attend_tc<D>, grid, dim3(kThreads), smem, st, 1, a);                         \
    if (e != cudaSuccess) return e;                                                               \
    break;
    CASE(128) CASE(256) CASE(384) CASE(512)
#undef CASE
    default: return cudaErrorInvalidValue;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess || a.n_splits == 1) return e;
  return launch_attend_combine(a, rows, st);
}

}  // namespace csa
