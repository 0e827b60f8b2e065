// Device-side helpers shared by the kernels of the CSA/HCA library (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/csa.h"

namespace csa {

// Geometry + pointers of one cache, passed to kernels by value.
struct CacheView {
  int m, d, d_rope, d_idx, kv_dtype, win_dtype, n_win, win_cap, page_size, max_pages;
  long long max_entries;
  long long cap;          // entry capacity per sequence
  const uint8_t *kv_nope;
  const float *kv_scale;
  const uint8_t *kv_rope;
  const uint8_t *idx_key;
  const float *idx_scale;
  const int32_t *page_table;
  const uint8_t *win;
  float *pool_state;
  long long *n_tokens;
  int idx_fp4;            // indexer keys are packed e2m1 (two per byte) + per-entry scale
};

// Per-frequency phase increments of the rotary embedding, as 64-bit fixed-point
// fractions of a turn: step[i] = round(2^64 * theta^(-2i/d_rope) / (2*pi)).
// Position p turns pair i by (p * step[i] mod 2^64) / 2^64 of a full turn, which
// is exact integer arithmetic for any p; only the final sin/cos is in fp32.
struct RopeTable {
  unsigned long long step[32];
};

__device__ __forceinline__ long long entry_row(const CacheView &c, int b, long long j) {
  if (c.page_size == 0) return (long long)b * c.max_entries + j;
  const int pg = __ldg(c.page_table + (long long)b * c.max_pages + j / c.page_size);
  return (long long)pg * c.page_size + j % c.page_size;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// e4m3 code -> float.  The code's 7 magnitude bits shifted into an fp16 pattern
// (exponent bias 15 instead of 7) give the value times 2^-8 exactly, subnormals
// included; the factor is undone in fp32.
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  const uint16_t h = (uint16_t)(((c & 0x80u) << 8) | ((c & 0x7Fu) << 7));
  return __half2float(__ushort_as_half(h)) * 256.0f;
}

// Two e4m3 codes (low bytes of v) -> two fp16 values that are the codes' values
// times 2^-8 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_scaled(uint32_t v) {
  // bytes b0 -> bits 15..8, b1 -> bits 31..24
  const uint32_t x = __byte_perm(v, 0u, 0x1404);   // [b1, 0, b0, 0] as bytes 3..0 -> 0x b1 00 b0 00
  return (x & 0x80008000u) | ((x & 0x7F007F00u) >> 1);
}

__device__ __forceinline__ uint8_t f32_to_e4m3_rn_sat(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// e2m1 (FP4) code of x, round to nearest with ties to the even code (mantissa bit 0),
// saturating at +-6; -0 and values that round to 0 give code 0.
__device__ __forceinline__ uint32_t f32_to_e2m1_rn_sat(float x) {
  const float a = fabsf(x);
  const uint32_t m = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) + (uint32_t)(a >= 1.75f) +
                     (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) + (uint32_t)(a > 5.0f);
  return m | ((x < 0.f && m) ? 8u : 0u);
}

// e2m1 code (low 4 bits) -> float
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
  const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  const float v = mag[c & 7u];
  return (c & 8u) ? -v : v;
}

// Eight packed e2m1 codes (a 32-bit word, code k in bits 4k..4k+3) -> eight e4m3 codes
// of the same values (exact: every e2m1 value is an e4m3 value), bytes k of {lo, hi}.
__device__ __forceinline__ void e2m1x8_to_e4m3x8(uint32_t w, uint32_t &lo, uint32_t &hi) {
  constexpr uint32_t kMagLo = 0x3C383000u, kMagHi = 0x4C484440u;   // e4m3 of 0, .5, 1, 1.5 | 2, 3, 4, 6
  const uint32_t s = (w >> 3) & 0x11111111u;                        // sign of each code, one bit per nibble
  lo = __byte_perm(kMagLo, kMagHi, w & 0x7777u) | __byte_perm(0x8000u, 0u, s & 0xFFFFu);
  hi = __byte_perm(kMagLo, kMagHi, (w >> 16) & 0x7777u) | __byte_perm(0x8000u, 0u, s >> 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// cos / sin of (pos * step / 2^64) turns.  The top 24 bits of the signed phase
// go through sincospif exactly; the remaining bits (< 2^-24 turn) enter as a
// first-order correction.
__device__ __forceinline__ void rope_cos_sin(long long pos, unsigned long long step, float &c, float &s) {
  const long long ph = (long long)((unsigned long long)pos * step);
  const long long top = ph >> 40;                                // [-2^23, 2^23)
  const long long rest = ph - (top << 40);                        // [0, 2^40)
  const float r_hi = (float)top * 0x1p-23f;                       // 2*turns, exact
  const float delta = (float)rest * 0x1p-64f * 6.28318530717958647692f;   // radians
  float sh, ch;
  sincospif(r_hi, &sh, &ch);
  c = ch - sh * delta;
  s = sh + ch * delta;
}

__device__ __forceinline__ float load_tok(const uint8_t *base, int dtype, long long i) {
  return dtype == CSA_F32 ? __ldg(reinterpret_cast<const float *>(base) + i)
                          : bf16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t *>(base) + i));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Order-preserving map float -> uint32 (larger float -> larger key); -0 and +0
// get the same key, as they compare equal.
__device__ __forceinline__ uint32_t float_key(float f) {
  const uint32_t u = f == 0.f ? 0u : __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Programmatic dependent launch (off unless built with -DCSA_PDL).  With it,
// kernels of one step are launched with programmatic stream serialization, so a
// kernel may start while its predecessor finishes.  pdl_wait() blocks until the
// predecessor grid has completed and its writes are visible; every kernel calls
// pdl_trigger() only after its own pdl_wait(), so code before pdl_wait() may read
// anything written two or more kernels earlier, never the direct predecessor's
// output.  Without it both are no-ops and stream order serialises the kernels.
#ifdef CSA_PDL
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#else
__device__ __forceinline__ void pdl_wait() {}
__device__ __forceinline__ void pdl_trigger() {}
#endif

// Device status word at the start of every workspace.
struct WsHeader {
  int status;
  int pad[63];
};

}  // namespace csa
