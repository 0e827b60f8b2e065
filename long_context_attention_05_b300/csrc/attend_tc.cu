// a4 / a5 — shared-KV multi-query attention on tensor cores (mma.sync f16).
//
// Sources: "DeepSeek V4 infrastructure" (volanea.com), "Compression only works
// if the attention path is engineered end to end" — shared key-value
// multi-query attention, partial RoPE, sliding-window branch, attention sink;
// "DeepSeek V4: How They Crushed the Million-Token Memory Problem"
// (sameershanbhag.com), "Two kinds of memory instead of one" — attention over
// the selected (CSA) or all (HCA) compressed entries plus the window.
//
// One CTA = one query row x a range of 64-key chunks, all heads (<= 64).
// Operands are f16:
//   q    : rotated at t in fp32, times a per-head power of two S_h (max|q|S_h < 2^14)
//   entry: e4m3 dims as code * 2^-8 (exact bit re-mapping), rotary dims bf16 -> f16
//   window token: raw bf16 -> f16, rotary dims turned at its position
// Logits: l = (sigma_j * S_nope + S_rope) / (S_h sqrt(d)) with sigma_j = 2^8 s_j for
// an entry (s_j its scale) and 1 for a window token; the e4m3 and rotary parts
// accumulate separately because they carry different scales.  Values: the same
// key rows (shared KV); the e4m3 dims use P' = P * sigma_j, the rotary dims P.
// P is stored in f16 (11 significant bits).
//
// 16 warps: in the logit phase warp (g, q) computes heads 16g.. x keys 16q..;
// the softmax runs on the 64x64 logit tile in shared memory; in the value phase
// warp (g, q) accumulates heads 16g.. x dims q*d/4 .. in registers.
#include "kernels.h"

namespace csa {
namespace {

constexpr int kKeys = 64;           // keys per chunk
constexpr int kHeadsMax = 64;
constexpr int kThreads = 512;
constexpr int kPadH = 8;            // f16 row padding (16 bytes) against bank conflicts

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void ldm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1) k_attend_tc(AttendArgs a) {
  constexpr int DN = D - 64;                 // e4m3 dims (rotary dims: the last 64)
  constexpr int LDQ = D + kPadH;             // f16 row stride of Q and K tiles
  constexpr int LDP = kKeys + kPadH;         // f16 row stride of P tiles
  constexpr int LDS = kKeys + 4;             // fp32 row stride of the logit tile
  constexpr int DQ = D / 4;                  // dims per warp in the value phase
  constexpr int NT = DQ / 8;                 // n-tiles per warp in the value phase
  constexpr int kGatherPer = (kKeys * ((D - 64) / 16 > D / 8 - 8 ? (D - 64) / 16 + 8 : D / 8) + kThreads - 1) / kThreads;
  extern __shared__ __align__(16) uint8_t smem[];
  __half *Qs = reinterpret_cast<__half *>(smem);                        // [64][LDQ]
  __half *Ks = Qs + kHeadsMax * LDQ;                                     // [64][LDQ]
  float *Sf = reinterpret_cast<float *>(Ks + kKeys * LDQ);              // [64][LDS]
  __half *Ph = reinterpret_cast<__half *>(Sf + kHeadsMax * LDS);        // [64][LDP]  P
  __half *Pn = Ph + kHeadsMax * LDP;                                     // [64][LDP]  P * sigma
  float *sig = reinterpret_cast<float *>(Pn + kHeadsMax * LDP);         // [64] sigma_j
  float *qsc = sig + kKeys;                                              // [64] 1/(S_h sqrt d)
  float *m_run = qsc + kHeadsMax;
  float *l_run = m_run + kHeadsMax;
  float *corr = l_run + kHeadsMax;
  long long *ksrc = reinterpret_cast<long long *>(corr + kHeadsMax);    // [64]
  float2 *qcs = reinterpret_cast<float2 *>(ksrc + kKeys);               // [32] (cos, sin) at t
  float2 *wcs = qcs + 32;                                                // [64][32] window tokens' (cos, sin)

  const CacheView &c = a.c;
  const int row = blockIdx.y;
  const int b = row / a.n_q, iq = row % a.n_q;
  const long long t = c.n_tokens[b] - a.n_q + iq;
  const long long n_vis = min((t + 1) / c.m, c.cap);
  const long long n_list = a.idx ? a.k : n_vis;
  const long long U = n_list + c.n_win;
  const int H = a.heads;
  const int split = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = warp & 3, qq = warp >> 2;
  // splits past this row's keys (the plan covers the key-list capacity) do nothing;
  // the merge reads only the splits that hold keys.  Only a dense (HCA) row can end
  // early: a selected list always has k slots, so a sparse row's check needs no
  // n_tokens and does not hold back the query loads below.
  if (a.idx == nullptr && a.n_splits > 1 && (long long)split * a.keys_per_split >= U) return;   // uniform

  // key source of slot tid of a chunk: entry row (>= 0), -2 - ring row (window
  // token; the ring slot is resolved here, once per key, not per gathered piece)
  // or -1 (no key); sigma as described above
  auto key_src = [&](long long u0) {
    const long long u = u0 + tid;
    long long src = -1;
    if (u < n_list) {
      const long long j = a.idx ? (long long)__ldg(a.idx + (long long)row * a.k + u) : u;
      if (j >= 0 && j < n_vis) src = entry_row(c, b, j);
    } else if (u < U) {
      const long long tau = t - c.n_win + 1 + (u - n_list);
      if (tau >= 0) src = -2 - ((long long)b * c.win_cap + tau % c.win_cap);
    }
    return src;
  };
  // ---- gather of a chunk's key tile as f16, in 16-byte pieces: gather_load issues
  //      every load of this thread into registers, gather_store converts and stores
  constexpr int NOPE16 = DN / 16;   // 16-byte e4m3 pieces per entry
  constexpr int ROPE16 = 64 / 8;    // 16-byte bf16 pieces of the rotary dims
  constexpr int RAW16 = D / 8;      // 16-byte bf16 pieces of a raw window token
  constexpr int PIECES = NOPE16 > RAW16 - ROPE16 ? NOPE16 + ROPE16 : RAW16;
  auto gather_load = [&](uint4 (&buf)[kGatherPer]) {
#pragma unroll
    for (int r = 0; r < kGatherPer; ++r) {
      const int x = tid + r * kThreads;
      buf[r] = make_uint4(0, 0, 0, 0);
      if (x < kKeys * PIECES) {
        const int kk = x / PIECES, p = x % PIECES;
        const long long src = ksrc[kk];
        if (src >= 0) {
          if (p < NOPE16) buf[r] = __ldg(reinterpret_cast<const uint4 *>(c.kv_nope + src * DN) + p);
          else if (p < NOPE16 + ROPE16)
            buf[r] = __ldg(reinterpret_cast<const uint4 *>(c.kv_rope + src * 64 * 2) + (p - NOPE16));
        } else if (src <= -2 && p < RAW16) {
          buf[r] = __ldg(reinterpret_cast<const uint4 *>(c.win + (-2 - src) * D * 2) + p);
        }
      }
    }
  };
  auto gather_store = [&](const uint4 (&buf)[kGatherPer]) {
#pragma unroll
    for (int r = 0; r < kGatherPer; ++r) {
      const int x = tid + r * kThreads;
      if (x >= kKeys * PIECES) continue;
      const int kk = x / PIECES, p = x % PIECES;
      const long long src = ksrc[kk];
      __half *dst = Ks + kk * LDQ;
      const uint4 u = buf[r];
      if (src >= 0) {
        if (p < NOPE16) {
          uint4 o0, o1;
          o0.x = e4m3x2_to_f16x2_scaled(u.x); o0.y = e4m3x2_to_f16x2_scaled(u.x >> 16);
          o0.z = e4m3x2_to_f16x2_scaled(u.y); o0.w = e4m3x2_to_f16x2_scaled(u.y >> 16);
          o1.x = e4m3x2_to_f16x2_scaled(u.z); o1.y = e4m3x2_to_f16x2_scaled(u.z >> 16);
          o1.z = e4m3x2_to_f16x2_scaled(u.w); o1.w = e4m3x2_to_f16x2_scaled(u.w >> 16);
          *reinterpret_cast<uint4 *>(dst + p * 16) = o0;
          *reinterpret_cast<uint4 *>(dst + p * 16 + 8) = o1;
        } else if (p < NOPE16 + ROPE16) {
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
          uint4 o;
          uint32_t *op = &o.x;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            op[e] = pack_h2(bf16_bits_to_f32((uint16_t)(w4[e] & 0xFFFF)), bf16_bits_to_f32((uint16_t)(w4[e] >> 16)));
          *reinterpret_cast<uint4 *>(dst + DN + (p - NOPE16) * 8) = o;
        }
      } else if (src <= -2) {
        if (p < RAW16) {
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
          float f[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            f[2 * e] = bf16_bits_to_f32((uint16_t)(w4[e] & 0xFFFF));
            f[2 * e + 1] = bf16_bits_to_f32((uint16_t)(w4[e] >> 16));
          }
          if (p * 8 >= DN) {   // rotary dims of a window token turn at its position
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const float2 cs = wcs[kk * 32 + ((p * 8 + e - DN) >> 1)];
              const float x0 = f[e], x1 = f[e + 1];
              f[e] = fmaf(x0, cs.x, -x1 * cs.y);
              f[e + 1] = fmaf(x0, cs.y, x1 * cs.x);
            }
          }
          uint4 o;
          o.x = pack_h2(f[0], f[1]); o.y = pack_h2(f[2], f[3]);
          o.z = pack_h2(f[4], f[5]); o.w = pack_h2(f[6], f[7]);
          *reinterpret_cast<uint4 *>(dst + p * 8) = o;
        }
      } else if (p < RAW16) {
        *reinterpret_cast<uint4 *>(dst + p * 8) = make_uint4(0, 0, 0, 0);
      }
    }
  };

  // (cos, sin) of every rotary pair of the chunk's window tokens, spread over all
  // threads (4 each) instead of falling on the few threads that hold rotary pieces
  auto win_rope = [&](long long u0) {
#pragma unroll
    for (int r = 0; r < kKeys * 32 / kThreads; ++r) {
      const int e = tid + r * kThreads, kk = e >> 5, pr = e & 31;
      if (ksrc[kk] <= -2) {
        const long long tau = t - c.n_win + 1 + (u0 + kk - n_list);   // the token's position
        float cs, sn;
        rope_cos_sin(tau, a.rope.step[pr], cs, sn);
        wcs[e] = make_float2(cs, sn);
      }
    }
  };

  const long long ch0 = (long long)split * a.chunks_per_split;
  constexpr int QH = kHeadsMax / (kThreads / 32);          // heads per warp
  constexpr int QV = (D / 32) % 8 == 0 ? (D / 32) / 8 : 1;  // 16-byte pieces per lane per head
  uint4 qraw[QH][QV];
  // prologue: every independent memory access of the first chunk goes out before
  // any conversion work -- the first chunk's key lookups, the query rows, then
  // (once the key rows are known) the key gather
  long long src_next = -1;
  float sig_next = 0.f, scale_first = 0.f;
  // the query rows and n_tokens are ready before this kernel starts; the key
  // indices come from the kernel just before it
  if (a.q_dtype == CSA_BF16 && (D / 32) % 8 == 0) {
#pragma unroll
    for (int hh = 0; hh < QH; ++hh) {
      const int h = warp + hh * (kThreads / 32);
#pragma unroll
      for (int u = 0; u < QV; ++u)
        qraw[hh][u] = h < H ? __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(a.q) +
                                                                     ((long long)row * H + h) * D + lane * (D / 32)) + u)
                            : make_uint4(0, 0, 0, 0);
    }
  }
  pdl_wait();
  pdl_trigger();
  if (tid < kKeys) {
    const long long src = ch0 * kKeys < U ? key_src(ch0 * kKeys) : -1;
    ksrc[tid] = src;
    if (src >= 0) scale_first = __ldg(c.kv_scale + src);   // consumed after the query work
    sig[tid] = src <= -2 ? 1.f : 0.f;
  }
  // ---- query: one (cos, sin) per rotary pair at t, shared by all heads
  if (tid < 32) {
    float cs, sn;
    rope_cos_sin(t, a.rope.step[tid], cs, sn);
    qcs[tid] = make_float2(cs, sn);
  }
  // warp w converts heads w, w+16, ...; lane holds D/32 consecutive dims (its
  // 16-byte query loads were issued at the top)
  __syncthreads();   // ksrc, qcs visible
  uint4 gbuf[kGatherPer];
  gather_load(gbuf);
  const bool win0 = ch0 * kKeys < U && ch0 * kKeys + kKeys > n_list;   // uniform: window tokens in chunk 0
  if (win0) win_rope(ch0 * kKeys);
  {
    // The heads of this warp go through each step together, QG at a time
    // (independent chains: a group costs the latency of one head, not of QG).
    constexpr int PER = D / 32;
    constexpr int QG = QH;
#pragma unroll
    for (int hg = 0; hg < QH; hg += QG) {
    float v[QG][PER];
#pragma unroll
    for (int hh = 0; hh < QG; ++hh) {
      const int h = warp + (hg + hh) * (kThreads / 32);
      if (h < H) {
        const long long q0 = ((long long)row * H + h) * D + lane * PER;
        if (a.q_dtype == CSA_BF16 && PER % 8 == 0) {   // from the 16-byte loads issued above
#pragma unroll
          for (int u = 0; u < PER / 8; ++u) {
            const uint4 x = qraw[hg + hh][u];
            const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              v[hh][u * 8 + 2 * e] = bf16_bits_to_f32((uint16_t)(w4[e] & 0xFFFF));
              v[hh][u * 8 + 2 * e + 1] = bf16_bits_to_f32((uint16_t)(w4[e] >> 16));
            }
          }
        } else if (a.q_dtype == CSA_BF16 && PER == 4) {   // d = 128: one 8-byte load
          const uint2 x = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(a.q) + q0));
          v[hh][0] = bf16_bits_to_f32((uint16_t)(x.x & 0xFFFF));
          v[hh][1] = bf16_bits_to_f32((uint16_t)(x.x >> 16));
          v[hh][2] = bf16_bits_to_f32((uint16_t)(x.y & 0xFFFF));
          v[hh][3] = bf16_bits_to_f32((uint16_t)(x.y >> 16));
        } else {
#pragma unroll
          for (int e = 0; e < PER; ++e) v[hh][e] = load_tok(a.q, a.q_dtype, q0 + e);
        }
      } else {
#pragma unroll
        for (int e = 0; e < PER; ++e) v[hh][e] = 0.f;
      }
    }
    // rotary turn of the pairs this lane holds (last 64 dims)
    if (lane * PER + PER > DN) {
#pragma unroll
      for (int e = 0; e < PER; e += 2) {
        const int dim = lane * PER + e;
        if (dim >= DN) {
          const float2 cs = qcs[(dim - DN) >> 1];
#pragma unroll
          for (int hh = 0; hh < QG; ++hh) {
            const float x0 = v[hh][e], x1 = v[hh][e + 1];
            v[hh][e] = fmaf(x0, cs.x, -x1 * cs.y);
            v[hh][e + 1] = fmaf(x0, cs.y, x1 * cs.x);
          }
        }
      }
    }
    float am[QG];
#pragma unroll
    for (int hh = 0; hh < QG; ++hh) {
      am[hh] = 0.f;
#pragma unroll
      for (int e = 0; e < PER; ++e) am[hh] = fmaxf(am[hh], fabsf(v[hh][e]));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
#pragma unroll
      for (int hh = 0; hh < QG; ++hh) am[hh] = fmaxf(am[hh], __shfl_xor_sync(0xffffffffu, am[hh], o));
    }
#pragma unroll
    for (int hh = 0; hh < QG; ++hh) {
      const int h = warp + (hg + hh) * (kThreads / 32);
      int ex = 0;
      frexpf(am[hh], &ex);
      const float S = am[hh] > 0.f ? ldexpf(1.f, 14 - ex) : 1.f;
      // 16-byte (or 8-byte) stores: a lane's PER halves are contiguous, and 4-byte
      // stores at a 2*PER-byte lane stride would conflict PER/2 ways
      uint32_t pk[PER / 2];
#pragma unroll
      for (int e = 0; e < PER; e += 2) pk[e / 2] = pack_h2(v[hh][e] * S, v[hh][e + 1] * S);
      if constexpr (PER % 8 == 0) {
        uint4 *dst = reinterpret_cast<uint4 *>(Qs + h * LDQ + lane * PER);
#pragma unroll
        for (int u = 0; u < PER / 8; ++u) dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      } else {
        uint2 *dst = reinterpret_cast<uint2 *>(Qs + h * LDQ + lane * PER);
#pragma unroll
        for (int u = 0; u < PER / 4; ++u) dst[u] = make_uint2(pk[2 * u], pk[2 * u + 1]);
      }
      if (lane == 0) {
        qsc[h] = a.scale / S;
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
      }
    }
    }
  }

  if (tid < kKeys) {
    if (ksrc[tid] >= 0) sig[tid] = 256.f * scale_first;
    // look up the next chunk's keys now; used one chunk later
    const long long u1 = (ch0 + 1) * kKeys;
    if (a.chunks_per_split > 1 && u1 < U) {
      src_next = key_src(u1);
      sig_next = src_next >= 0 ? 256.f * __ldg(c.kv_scale + src_next) : (src_next <= -2 ? 1.f : 0.f);
    }
  }
  if (win0) __syncthreads();   // window (cos, sin) table visible
  gather_store(gbuf);

  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[n][r] = 0.f;

  for (long long chunk = ch0; chunk < ch0 + a.chunks_per_split; ++chunk) {
    const long long u0 = chunk * kKeys;
    if (u0 >= U) break;
    __syncthreads();   // previous chunk's value phase is done with Ks / P (first chunk: its tile is stored)
    if (chunk != ch0) {
      if (tid < kKeys) {
        ksrc[tid] = src_next;
        sig[tid] = sig_next;
        const long long u1 = u0 + kKeys;
        src_next = -1;
        sig_next = 0.f;
        if (chunk + 1 < ch0 + a.chunks_per_split && u1 < U) {
          src_next = key_src(u1);
          sig_next = src_next >= 0 ? 256.f * __ldg(c.kv_scale + src_next) : (src_next <= -2 ? 1.f : 0.f);
        }
      }
      __syncthreads();
      gather_load(gbuf);
      if (u0 + kKeys > n_list) {   // uniform
        win_rope(u0);
        __syncthreads();
      }
      gather_store(gbuf);
      __syncthreads();
    }
    // ---- logits: warp (g, qq): heads 16g..16g+15 x keys 16qq..16qq+15
    if (16 * g < H) {
      // e4m3 part: two accumulator chains per n-tile (even / odd K steps) so the
      // dependent MMAs interleave; rotary part: one chain per n-tile
      float sn[2][4] = {}, sn2[2][4] = {}, sr[2][4] = {};
      const uint32_t qa = su32(Qs + (16 * g + (lane & 15)) * LDQ + (lane >> 4) * 8);
      const uint32_t kb = su32(Ks + (16 * qq + (lane & 7) + ((lane >> 4) << 3)) * LDQ + ((lane >> 3) & 1) * 8);
#pragma unroll 4
      for (int ks = 0; ks < DN / 16; ks += 2) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3, c0, c1, c2, c3, d0, d1, d2, d3;
        ldm_x4(qa + ks * 32, a0, a1, a2, a3);
        ldm_x4(kb + ks * 32, b0, b1, b2, b3);
        ldm_x4(qa + ks * 32 + 32, c0, c1, c2, c3);
        ldm_x4(kb + ks * 32 + 32, d0, d1, d2, d3);
        mma16816(sn[0], a0, a1, a2, a3, b0, b1);
        mma16816(sn[1], a0, a1, a2, a3, b2, b3);
        mma16816(sn2[0], c0, c1, c2, c3, d0, d1);
        mma16816(sn2[1], c0, c1, c2, c3, d2, d3);
      }
#pragma unroll
      for (int ks = DN / 16; ks < D / 16; ++ks) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldm_x4(qa + ks * 32, a0, a1, a2, a3);
        ldm_x4(kb + ks * 32, b0, b1, b2, b3);
        mma16816(sr[0], a0, a1, a2, a3, b0, b1);
        mma16816(sr[1], a0, a1, a2, a3, b2, b3);
      }
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int r = 0; r < 4; ++r) sn[n][r] += sn2[n][r];
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int h = 16 * g + (lane >> 2) + (r >= 2 ? 8 : 0);
          const int kk = 16 * qq + 8 * n + 2 * (lane & 3) + (r & 1);
          Sf[h * LDS + kk] = ksrc[kk] != -1 ? (sig[kk] * sn[n][r] + sr[n][r]) * qsc[h] : -INFINITY;
        }
    }
    __syncthreads();
    // ---- online softmax: 8 threads per head, 8 keys each
    {
      const int h = tid >> 3, part = tid & 7;
      float sv[8];
      float cmax = -INFINITY;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        sv[e] = Sf[h * LDS + part * 8 + e];
        cmax = fmaxf(cmax, sv[e]);
      }
#pragma unroll
      for (int o = 4; o; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
      const float m_old = m_run[h];
      const float m_new = fmaxf(m_old, cmax);
      float psum = 0.f;
      uint32_t ph[4], pn[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const float p0 = (m_new > -INFINITY && sv[e] > -INFINITY) ? __expf(sv[e] - m_new) : 0.f;
        const float p1 = (m_new > -INFINITY && sv[e + 1] > -INFINITY) ? __expf(sv[e + 1] - m_new) : 0.f;
        psum += p0 + p1;
        ph[e / 2] = pack_h2(p0, p1);
        pn[e / 2] = pack_h2(p0 * sig[part * 8 + e], p1 * sig[part * 8 + e + 1]);
      }
#pragma unroll
      for (int o = 4; o; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      *reinterpret_cast<uint4 *>(Ph + h * LDP + part * 8) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
      *reinterpret_cast<uint4 *>(Pn + h * LDP + part * 8) = make_uint4(pn[0], pn[1], pn[2], pn[3]);
      __syncwarp();
      if (part == 0) {
        const float cr = m_old > -INFINITY ? __expf(m_old - m_new) : (m_new > -INFINITY ? 0.f : 1.f);
        corr[h] = cr;
        l_run[h] = l_run[h] * cr + psum;
        m_run[h] = m_new;
      }
    }
    __syncthreads();
    // ---- values: warp (g, qq): heads 16g.. x dims qq*DQ .. qq*DQ + DQ - 1
    if (16 * g < H) {
      const float c_lo = corr[16 * g + (lane >> 2)], c_hi = corr[16 * g + (lane >> 2) + 8];
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        acc[n][0] *= c_lo; acc[n][1] *= c_lo;
        acc[n][2] *= c_hi; acc[n][3] *= c_hi;
      }
      const uint32_t pa_off = ((16 * g + (lane & 15)) * LDP + (lane >> 4) * 8) * 2;
      const uint32_t pha = su32(Ph) + pa_off, pna = su32(Pn) + pa_off;
#pragma unroll
      for (int ks = 0; ks < kKeys / 16; ++ks) {
        uint32_t h0, h1, h2, h3, n0, n1, n2, n3;
        ldm_x4(pha + ks * 32, h0, h1, h2, h3);
        ldm_x4(pna + ks * 32, n0, n1, n2, n3);
        const uint32_t vb = su32(Ks + (ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LDQ + qq * DQ + (lane >> 4) * 8);
#pragma unroll
        for (int n = 0; n < NT; n += 2) {
          uint32_t b0, b1, b2, b3;
          ldm_x4_t(vb + n * 16, b0, b1, b2, b3);
          const bool nope0 = qq * DQ + n * 8 < DN, nope1 = qq * DQ + (n + 1) * 8 < DN;
          if (nope0) mma16816(acc[n], n0, n1, n2, n3, b0, b1);
          else mma16816(acc[n], h0, h1, h2, h3, b0, b1);
          if (nope1) mma16816(acc[n + 1], n0, n1, n2, n3, b2, b3);
          else mma16816(acc[n + 1], h0, h1, h2, h3, b2, b3);
        }
      }
    }
  }
  __syncthreads();
  // ---- output: finished rows (one split) or partials
  if (16 * g < H) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int h = 16 * g + (lane >> 2) + 8 * half;
      if (h >= H) continue;
      float f = 1.f, lse = 0.f;
      if (a.n_splits == 1) {
        const float z = __ldg(a.sink + h);
        const float mr = m_run[h];
        const float M = fmaxf(mr, z);
        const float em = mr > -INFINITY ? expf(mr - M) : 0.f;
        const float L = l_run[h] * em + expf(z - M);
        f = em / L;
        lse = M + logf(L);
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int dim = qq * DQ + n * 8 + 2 * (lane & 3);
        const float o0 = acc[n][2 * half] * f, o1 = acc[n][2 * half + 1] * f;
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
      if ((lane & 3) == 0 && qq == 0) {
        if (a.n_splits == 1) {
          if (a.out_lse) a.out_lse[(long long)row * H + h] = lse;
        } else {
          const long long pb = ((long long)row * a.n_splits + split) * H + h;
          a.part_ml[pb * 2] = m_run[h];
          a.part_ml[pb * 2 + 1] = l_run[h];
        }
      }
    }
  }
}

}  // namespace

bool attend_tc_supported(const CacheView &c, int heads, int q_dtype) {
  return c.kv_dtype == CSA_E4M3 && c.win_dtype == CSA_BF16 && c.d_rope == 64 &&
         (c.d == 128 || c.d == 256 || c.d == 384 || c.d == 512) && heads % 16 == 0 && heads <= kHeadsMax &&
         (q_dtype == CSA_BF16 || q_dtype == CSA_F32);
}

size_t attend_tc_smem_bytes(int d) {
  return (size_t)(2 * kHeadsMax * (d + kPadH)) * 2 + (size_t)kHeadsMax * (kKeys + 4) * 4 +
         (size_t)2 * kHeadsMax * (kKeys + kPadH) * 2 + (size_t)(kKeys + 4 * kHeadsMax) * 4 + kKeys * 8 + 32 * 8 +
         (size_t)kKeys * 32 * 8;
}

cudaError_t launch_attend_tc(const AttendArgs &a, int rows, cudaStream_t st) {
  const size_t smem = attend_tc_smem_bytes(a.c.d);
  dim3 grid(a.n_splits, rows);
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
