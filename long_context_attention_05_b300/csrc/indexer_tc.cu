// a2 — lightning-indexer scoring on the 5th-generation tensor cores (sm_103a).
//
// Sources: "DeepSeek V4: How They Crushed the Million-Token Memory Problem"
// (sameershanbhag.com), "Two kinds of memory instead of one" — a low-precision
// lightning indexer scores every compressed block with ReLU multi-head dot
// products and keeps the top-k; "DeepSeek V4 infrastructure" (volanea.com),
// "Compression only works if the attention path is engineered end to end" — a
// selector whose scoring path burns memory bandwidth becomes the bottleneck.
//
// score_j = s_j * sum_h w_h * ReLU(q_h . code_j)  (s_j > 0 is the key's scale).
//
// Design.  The e4m3 keys stream from HBM once, by TMA, straight into the tensor
// cores: D[entry, head] = sum_k code[entry, k] * q'[head, k] with
// tcgen05.mma kind::f8f6f4, M = 128 entries (one TMEM lane each), N = 2 x heads
// (the hi and lo query operands stacked), K = 128 (four K=32 steps over one
// 128-byte swizzled row).  The bf16 query is
// made an exact pair of e4m3 operands: per head a power of two S_h puts
// max|q_h| below 2^8, hi = e4m3(q*S_h), lo = e4m3((q*S_h - hi) * 16); for every
// component with |q*S_h| >= 2^-6 this is exact (8 significant bits = 4 + 4), so
// the product q . code is the bf16 query's product up to fp32 accumulation.
// Per tile one accumulator of 2*heads columns (hi | lo); up to four in TMEM.
// The epilogue thread of TMEM lane l owns entry l of the tile:
//   score = s_j * sum_h (w_h / S_h) * ReLU(D_hi[h] + D_lo[h] / 16).
//
// Warp roles (448 threads): warp 0 = TMA producer, warp 1 = MMA issuer and TMEM
// owner, warps 2..13 = three epilogue warpgroups that take tiles in turn (warp w
// reads TMEM lane group w % 4).  Pipelines: an 8-stage shared-memory ring of key
// tiles (full/empty mbarriers) and up to four TMEM accumulator buffers
// (tmem_full/tmem_empty).  Every wait is bounded; a
// timeout sets the workspace status word and all roles stop issuing work.
// Each CTA scores a contiguous range of 128-entry tiles of one query row, so its
// query operand is built once (see the work assignment at the top of the kernel).
// Given per-row histograms (the fused index + top-k call), the epilogue also counts
// every score by the top kPrefixBits bits of its order-preserving key, in shared
// memory, and adds the counts to the row's histogram at the end.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.h"

namespace csa {
namespace {

constexpr int kTileM = 128;
constexpr int kDI = 128;
constexpr int kStages = 8;
constexpr int kStageBytes = kTileM * kDI;
constexpr int kEpiGroups = 3;   // epilogue warpgroups; group e takes tiles it % 3 == e
constexpr int kThreads = 64 + 128 * kEpiGroups;
constexpr int kMaxFlatRows = 256;   // the flat grid serves fewer query rows than this
// FP4 keys: TMA brings packed rows (64 bytes per entry) into kStages raw stages of
// 8 KB; a converter warpgroup turns each into a 16 KB e4m3 tile (the same 128-byte
// swizzled layout TMA gives e4m3 keys) in one of kConvStages stages that the MMA
// reads.  Both rings fit in the 128 KB the e4m3 key ring uses.
constexpr int kConvStages = 4;
constexpr int kRawStageBytes = kTileM * kDI / 2;

struct TcArgs {
  CacheView c;
  int n_q, heads, q_dtype;
  const uint8_t *q_idx;
  const float *w;
  float *scores;
  long long stride;
  int ctas_per_row;   // > 0: grid (ctas_per_row, rows); 0: flat grid, proportional split
  int rows;           // query rows (batch * n_q)
  int grid_sms;       // G of the proportional split
  int box_rows;       // rows per TMA box: 128 (contiguous) or the page size
  int *status;        // workspace status word (may be null)
  long long wait_limit;   // polls before a bounded wait gives up
  int starve;         // failure injection for tests: the producer issues no key copies
  int q_vec;          // q_idx is 16-byte aligned: vector loads of the query
  int hi_only;        // query-side FP8 variant: one e4m3 operand (N = heads), no lo term
  int fp4;            // FP4 keys: raw ring + converter warpgroup (the last epilogue group)
  unsigned *hist;     // per-row histograms of score-key prefixes (kPrefixBins each), or null
  unsigned *sel_ctr;  // the row-split top-k's per-row counters and digit counts, zeroed here, or null
  int sel_ctr_words;
};

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of `parity` to complete.  Gives up (returning
// false) when another role has aborted or after `limit` polls, in which case
// it raises the abort flag and records CSA_ERR_TIMEOUT.
__device__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *status, long long limit) {
  for (long long i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63 && *abort_flag) return false;
  }
  *abort_flag = 1;
  if (status) atomicExch(status, CSA_ERR_TIMEOUT);
  return false;
}

// Key tiles are read once per call: they go through L2 with the evict-first policy,
// so the stream does not push out what the next kernels reuse (scores, queries,
// window, code).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(su32(dst)),
      "l"((uint64_t)map), "r"(su32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// atoms 1024 bytes apart (sm_100 descriptor format, version 1).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

#define CSA_R8(i) "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), "=r"(v[i + 4]), "=r"(v[i + 5]), \
                  "=r"(v[i + 6]), "=r"(v[i + 7])
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : CSA_R8(0), CSA_R8(8), CSA_R8(16), CSA_R8(24)
      : "r"(taddr));
}
#undef CSA_R8
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads, 1) k_index_tc(const __grid_constant__ CUtensorMap kmap, TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t *stage = base;                                   // kStages x 16 KB key tiles
  uint8_t *bhi = base + kStages * kStageBytes;             // [heads][128] e4m3 hi, swizzled
  uint8_t *blo = bhi + a.heads * kDI;                      // [heads][128] e4m3 lo, right after:
                                                           // one N = 2*heads operand
  float *wq = reinterpret_cast<float *>(bhi + 2 * 128 * kDI);  // [heads] w_h / S_h
  uint64_t *full = reinterpret_cast<uint64_t *>(wq + 128);
  uint64_t *empty = full + kStages;
  uint64_t *tfull = empty + kStages;
  uint64_t *tempty = tfull + 4;
  uint64_t *cfull = tempty + 4;    // FP4: converted tile ready (4 converter warps)
  uint64_t *cempty = cfull + kConvStages;   // FP4: converted tile consumed (MMA commit)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(cempty + kConvStages);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  uint64_t *drain = cempty + kConvStages + 1;   // MMA drain after an abort (the 8 bytes after tmem_slot, abort_flag)
  unsigned *shist = reinterpret_cast<unsigned *>(reinterpret_cast<uint8_t *>(cempty + kConvStages) + 16);   // [kPrefixBins]
  // FP4: the e4m3 tiles the MMA reads are stage[0 .. kConvStages) (16 KB each); the raw
  // packed tiles TMA writes follow them, kStages x 8 KB
  uint8_t *raw = base + kConvStages * kStageBytes;

  const CacheView &c = a.c;
  // ---- work assignment.  Many query rows (>= one per SM): CTA y takes row y.
  // Few rows: the grid is flat (one CTA per SM) and row r gets ceil(tiles_r / L) CTAs
  // for the smallest per-CTA tile load L that fits the grid, so ragged context lengths
  // stay balanced; every CTA derives the same partition from n_tokens.
  __shared__ int sh_row, sh_sub, sh_cnt;
  __shared__ long long sh_nvis;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();      // n_tokens comes from the compressor just before
  pdl_trigger();
  if (threadIdx.x == 32) {   // barriers (warp 1) while warp 0 works out the partition
    // full/empty guard the TMA ring (e4m3 tiles, or FP4 raw tiles whose consumers are
    // the 4 converter warps); cfull/cempty the converted FP4 tiles
    for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], a.fp4 ? 4 : 1); }
    for (int s = 0; s < kConvStages; ++s) { mbar_init(&cfull[s], 4); mbar_init(&cempty[s], 1); }
    for (int s = 0; s < 4; ++s) { mbar_init(&tfull[s], 1); mbar_init(&tempty[s], 4); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  auto visible = [&](long long n_tok, int r) {   // entries query row r sees
    return min((n_tok - a.n_q + r % a.n_q + 1) / c.m, c.cap);
  };
  if (a.hist)
    for (int e = threadIdx.x; e < kPrefixBins; e += kThreads) shist[e] = 0u;
  // the top-k that follows counts its CTAs and digits per row from zero (the previous
  // call's top-k has completed: it ran before this kernel's predecessor)
  if (a.sel_ctr) {
    const int cta = blockIdx.y * gridDim.x + blockIdx.x, n_cta = gridDim.x * gridDim.y;
    for (int e = cta * kThreads + threadIdx.x; e < a.sel_ctr_words; e += n_cta * kThreads) a.sel_ctr[e] = 0u;
  }
  if (a.ctas_per_row > 0) {
    if (threadIdx.x == 0) {
      sh_row = blockIdx.y; sh_sub = blockIdx.x; sh_cnt = a.ctas_per_row;
      sh_nvis = visible(c.n_tokens[blockIdx.y / a.n_q], blockIdx.y);
    }
  } else if (warp == 0) {
    // lane l holds rows l, l+32, ...: every n_tokens load is issued before the first
    // is used (one memory round trip); the rest is a few 32-bit shuffles per chunk of
    // 32 rows (this runs on one warp at the start of every CTA, so it is kept short)
    const int rows = gridDim.y == 1 ? a.rows : 0;
    const int n_chunks = (rows + 31) >> 5;
    long long nt[kMaxFlatRows / 32];
#pragma unroll
    for (int u = 0; u < kMaxFlatRows / 32; ++u) {
      const int r = lane + 32 * u;
      nt[u] = r < rows ? c.n_tokens[r / a.n_q] : 0;
    }
    long long nv[kMaxFlatRows / 32];
    int tiles[kMaxFlatRows / 32];
    long long T = 0;
#pragma unroll
    for (int u = 0; u < kMaxFlatRows / 32; ++u) {
      if (u >= n_chunks) break;   // warp-uniform
      const int r = lane + 32 * u;
      nv[u] = r < rows ? visible(nt[u], r) : 0;
      tiles[u] = nv[u] > 0 ? (int)((nv[u] + kTileM - 1) / kTileM) : 0;
      T += tiles[u];
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) T += __shfl_xor_sync(0xffffffffu, T, o);
    // Row r gets ceil(tiles_r / L) CTAs for the smallest tile load L that fits the
    // grid: L lies in [ceil(T/G), ceil(T/(G-rows))] (the upper end always fits,
    // since sum ceil(t/L) <= T/L + rows), found by bisection; equal rows settle at
    // the lower end on the first probe.
    const long long G = a.grid_sms;
    auto ctas_needed = [&](long long L) -> long long {
      long long need = 0;
#pragma unroll
      for (int u = 0; u < kMaxFlatRows / 32; ++u) {
        if (u >= n_chunks) break;   // warp-uniform
        need += (tiles[u] + L - 1) / L;
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) need += __shfl_xor_sync(0xffffffffu, need, o);
      return need;
    };
    long long Llo = max(1LL, (T + G - 1) / G), Lhi = max(Llo, (T + (G - rows) - 1) / max(G - rows, 1LL));
    if (ctas_needed(Llo) <= G) Lhi = Llo;
    while (Llo < Lhi) {   // warp-uniform
      const long long mid = (Llo + Lhi) >> 1;
      if (ctas_needed(mid) <= G) Lhi = mid; else Llo = mid + 1;
    }
    const long long L = Lhi;
    int found_row = -1, found_sub = 0, found_cnt = 0, base = 0;
    long long found_nv = 0;
#pragma unroll
    for (int u = 0; u < kMaxFlatRows / 32; ++u) {
      if (u >= n_chunks) break;   // warp-uniform
      const int r = lane + 32 * u;
      const int cr = (int)((tiles[u] + L - 1) / L);
      int incl = cr;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int start = base + incl - cr;
      const bool mine = cr > 0 && (int)blockIdx.x >= start && (int)blockIdx.x < start + cr;
      const unsigned who = __ballot_sync(0xffffffffu, mine);
      if (who && found_row < 0) {
        const int src = __ffs(who) - 1;
        found_row = __shfl_sync(0xffffffffu, r, src);
        found_sub = (int)blockIdx.x - __shfl_sync(0xffffffffu, start, src);
        found_cnt = __shfl_sync(0xffffffffu, cr, src);
        found_nv = __shfl_sync(0xffffffffu, nv[u], src);
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) { sh_row = found_row; sh_sub = found_sub; sh_cnt = found_cnt; sh_nvis = found_nv; }
  }
  __syncthreads();
  if (sh_row < 0) return;   // uniform: a spare CTA of the flat grid
  const int row = sh_row;
  const int b = row / a.n_q;
  const long long n_vis = sh_nvis;
  const long long n_tiles = (n_vis + kTileM - 1) / kTileM;
  const long long tile_lo = (long long)sh_sub * n_tiles / sh_cnt;
  const long long tile_hi = (long long)(sh_sub + 1) * n_tiles / sh_cnt;
  if (tile_lo >= tile_hi) return;   // uniform: nothing allocated yet
  const int n_it = (int)(tile_hi - tile_lo);
  const int H = a.heads;
  const int n_acc = H <= 64 ? 4 : 2;                        // accumulator buffers (2H columns each)
  const uint32_t ncols = H <= 32 ? 256u : 512u;
  uint32_t tmem = 0;
  int issued = 0;   // key copies the producer issued (lane 0 of warp 0)
  if (warp != 0) {
    if (warp == 1) {   // TMEM first: it does not depend on the query
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                   "r"(ncols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // ---- query operand (warps 1.., while warp 0 already streams keys): per-head
    //      power-of-two scale, exact e4m3 hi/lo split, written in the K-major
    //      128-byte-swizzle layout the MMA reads.  Warp w builds heads w-1, w-1+13, ...;
    //      all of its query and weight loads are issued before the first is used, so
    //      the build costs one memory round trip (the key stream keeps HBM queues full
    //      by then, and a round trip per head added microseconds to every CTA's start).
    constexpr int kQW = kThreads / 32 - 1;           // builder warps
    constexpr int kMaxHPW = (128 + kQW - 1) / kQW;   // heads per builder warp (H <= 128)
    const int w0 = warp - 1;
    float4 qv[kMaxHPW];
#pragma unroll
    for (int u = 0; u < kMaxHPW; ++u) {
      const int h = w0 + u * kQW;
      qv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (h < H) {
        const long long q0 = ((long long)row * H + h) * kDI + lane * 4;
        if (a.q_vec && a.q_dtype == CSA_BF16) {
          const uint2 r = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(a.q_idx) + q0));
          qv[u] = make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xFFFF0000u),
                              __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xFFFF0000u));
        } else if (a.q_vec) {
          qv[u] = __ldg(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(a.q_idx) + q0));
        } else {
          qv[u] = make_float4(load_tok(a.q_idx, a.q_dtype, q0), load_tok(a.q_idx, a.q_dtype, q0 + 1),
                              load_tok(a.q_idx, a.q_dtype, q0 + 2), load_tok(a.q_idx, a.q_dtype, q0 + 3));
        }
      }
    }
    const float wl = (lane < kMaxHPW && w0 + lane * kQW < H) ? __ldg(a.w + (long long)row * H + w0 + lane * kQW) : 0.f;
    // loads issued: let the producer start the key stream (these small loads are then
    // ahead of it in the memory queues instead of behind megabytes of key tiles)
    asm volatile("bar.arrive 2, %0;" ::"n"(kThreads) : "memory");
    // the heads of this warp go through each step together (independent chains), so
    // the build's latency is that of one head, not of one head per step
    float am[kMaxHPW];
#pragma unroll
    for (int u = 0; u < kMaxHPW; ++u)
      am[u] = fmaxf(fmaxf(fabsf(qv[u].x), fabsf(qv[u].y)), fmaxf(fabsf(qv[u].z), fabsf(qv[u].w)));
#pragma unroll
    for (int o = 16; o; o >>= 1) {
#pragma unroll
      for (int u = 0; u < kMaxHPW; ++u) am[u] = fmaxf(am[u], __shfl_xor_sync(0xffffffffu, am[u], o));
    }
#pragma unroll
    for (int u = 0; u < kMaxHPW; ++u) {
      const int h = w0 + u * kQW;
      int ex = 0;
      frexpf(am[u], &ex);
      const float S = am[u] > 0.f ? ldexpf(1.f, 8 - ex) : 1.f;   // amax * S < 2^8
      const float v[4] = {qv[u].x, qv[u].y, qv[u].z, qv[u].w};
      uint32_t hw = 0, lw = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x = v[e] * S;
        const uint8_t hi = f32_to_e4m3_rn_sat(x);
        const uint8_t lo = a.hi_only ? (uint8_t)0 : f32_to_e4m3_rn_sat((x - e4m3_to_f32(hi)) * 16.f);
        hw |= (uint32_t)hi << (8 * e);
        lw |= (uint32_t)lo << (8 * e);
      }
      const float wh = __shfl_sync(0xffffffffu, wl, u);
      if (h < H) {
        const int k = lane * 4;   // 4 consecutive K bytes, inside one 16-byte chunk
        const int off = h * kDI + ((((k >> 4) ^ (h & 7)) << 4) | (k & 15));
        *reinterpret_cast<uint32_t *>(bhi + off) = hw;
        *reinterpret_cast<uint32_t *>(blo + off) = lw;
        if (lane == 0) wq[h] = wh / S;
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic-proxy writes -> tensor core reads
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads - 32) : "memory");   // all warps but the producer
    tc_fence_after();
    tmem = *tmem_slot;
  }

  if (warp == 0) {
    asm volatile("bar.sync 2, %0;" ::"n"(kThreads) : "memory");   // query loads are in flight
    {   // ---- TMA producer: lane 0 issues; for paged caches the whole warp keeps the
        //      page ids of the next 32 logical pages in flight (lane l holds page
        //      base + l), so no copy waits on a page-table load
      const uint64_t policy = l2_evict_first_policy();
      const int *ptab = c.page_size ? c.page_table + (long long)b * c.max_pages : nullptr;
      auto page_chunk = [&](long long base) -> int {   // page id of logical page base + lane
        const long long lp = base + lane;
        return (ptab && lp < c.max_pages) ? __ldg(ptab + lp) : 0;
      };
      long long pbase = -1;
      int pcur = 0, pnext = 0;
      for (int it = 0; it < (a.starve ? 0 : n_it); ++it) {
        const int s = it % kStages;
        const uint32_t ph = (uint32_t)(it / kStages) & 1u;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[s], ph ^ 1u, abort_flag, a.status, a.wait_limit);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;   // warp-uniform
        // e4m3 keys: 128-byte rows straight into the MMA's tile; FP4: 64-byte packed rows
        // into the raw ring
        const int row_bytes = a.fp4 ? kDI / 2 : kDI;
        uint8_t *dst = a.fp4 ? raw + s * kRawStageBytes : stage + s * kStageBytes;
        if (lane == 0) mbar_expect_tx(&full[s], kTileM * row_bytes);
        const long long tile = tile_lo + it;
        if (c.page_size == 0) {
          if (lane == 0)
            tma_load_2d(dst, &kmap, &full[s], 0, (int)((long long)b * c.max_entries + tile * kTileM), policy);
        } else {
          for (int r0 = 0; r0 < kTileM; r0 += a.box_rows) {
            const long long j0 = tile * kTileM + r0;
            const long long lp = j0 / c.page_size;   // past the table: page id 0 (never scored)
            if (pbase < 0 || lp >= pbase + 64) {     // (re)start: this chunk and the next
              pbase = lp;
              pcur = page_chunk(pbase);
              pnext = page_chunk(pbase + 32);
            } else if (lp >= pbase + 32) {            // next chunk: its ids are here, fetch the one after
              pbase += 32;
              pcur = pnext;
              pnext = page_chunk(pbase + 32);
            }
            const int pg = __shfl_sync(0xffffffffu, pcur, (int)(lp - pbase));
            if (lane == 0)
              tma_load_2d(dst + r0 * row_bytes, &kmap, &full[s], 0,
                          (int)((long long)pg * c.page_size + j0 % c.page_size), policy);
          }
        }
        ++issued;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {   // ---- MMA issuer
      // one MMA per K step: N = 2H columns, hi heads in [0, H), lo heads in [H, 2H)
      const int n_mma = a.hi_only ? H : 2 * H;   // hi only, or hi | lo
      const uint32_t idesc = (1u << 4) | ((uint32_t)(n_mma >> 3) << 17) | ((uint32_t)(kTileM >> 4) << 24);
      const uint32_t bh = su32(bhi);
      // the key tile: the TMA ring's stage (e4m3 keys) or the converted stage (FP4 keys)
      const int n_ring = a.fp4 ? kConvStages : kStages;
      uint64_t *tile_full = a.fp4 ? cfull : full, *tile_empty = a.fp4 ? cempty : empty;
      for (int it = 0; it < n_it; ++it) {
        const int s = it % n_ring;
        const uint32_t ph = (uint32_t)(it / n_ring) & 1u;
        const int acc = it % n_acc;
        const uint32_t aph = (uint32_t)(it / n_acc) & 1u;
        if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, a.status, a.wait_limit)) break;
        if (!mbar_wait(&tile_full[s], ph, abort_flag, a.status, a.wait_limit)) break;
        tc_fence_after();
        const uint32_t as = su32(stage + s * kStageBytes);
        const uint32_t d = tmem + (uint32_t)(acc * 2 * H);
#pragma unroll
        for (int kk = 0; kk < kDI / 32; ++kk)
          umma_f8(d, sw128_desc(as + kk * 32), sw128_desc(bh + kk * 32), idesc, kk > 0);
        umma_commit(&tile_empty[s]);
        umma_commit(&tfull[acc]);
      }
    }
  } else {   // ---- epilogue: TMEM lane group g = warp % 4 owns entries 32g .. 32g+31 of a tile
    const int g = warp & 3;
    // Groups take tiles in turn.  A group waits on an accumulator's next phase only
    // after finishing its previous tile, so the accumulator's previous use must be
    // older than that tile (parity waits would alias otherwise): groups <= buffers.
    const int n_grp = min(a.fp4 ? kEpiGroups - 1 : kEpiGroups, n_acc);   // FP4: the last group converts
    const int grp = (warp - 2) >> 2;   // epilogue group: tiles it with it % n_grp == grp
    // key scales are read four of this group's tiles ahead so their memory
    // latency overlaps the tiles in between instead of stalling each epilogue
    // paged caches: the page id of an entry is loaded one prefetch rotation before its
    // scale, so neither load waits on the other inside a tile's epilogue
    auto page_of = [&](int it2) -> int {
      const long long j2 = (tile_lo + it2) * kTileM + g * 32 + lane;
      return (c.page_size && it2 < n_it && j2 < n_vis)
                 ? __ldg(c.page_table + (long long)b * c.max_pages + j2 / c.page_size) : 0;
    };
    auto scale_of = [&](int it2, int pg) -> float {
      const long long j2 = (tile_lo + it2) * kTileM + g * 32 + lane;
      if (!(it2 < n_it && j2 < n_vis)) return 0.f;
      const long long r = c.page_size ? (long long)pg * c.page_size + j2 % c.page_size : (long long)b * c.max_entries + j2;
      return __ldg(c.idx_scale + r);
    };
    // slot u of sc[] holds the scale of this group's tile it0 + n_grp*u (pgn[u]: the page
    // id for the tile four group-tiles later); both are refilled in place
    float sc[4];
    int pgn[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) pgn[u] = page_of(grp + n_grp * u);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      sc[u] = scale_of(grp + n_grp * u, pgn[u]);
      pgn[u] = page_of(grp + n_grp * (u + 4));
    }
    bool live = true;
    if (grp >= n_grp) live = false;
    if (a.fp4 && grp == kEpiGroups - 1) {
      // ---- FP4 converter: thread = entry row r of the tile.  The 64 packed bytes of the
      //      row become its 128 e4m3 bytes, written in the 128-byte swizzle the MMA's
      //      descriptor expects (16-byte chunk j of row r at chunk j ^ (r & 7)).
      const int r = (warp - 2 - 4 * grp) * 32 + lane;
      for (int it = 0; it < n_it; ++it) {
        const int s = it % kStages, sc2 = it % kConvStages;
        const uint32_t ph = (uint32_t)(it / kStages) & 1u, pc = (uint32_t)(it / kConvStages) & 1u;
        bool ok = mbar_wait(&full[s], ph, abort_flag, a.status, a.wait_limit);
        if (ok) ok = mbar_wait(&cempty[sc2], pc ^ 1u, abort_flag, a.status, a.wait_limit);
        if (!__all_sync(0xffffffffu, ok)) break;   // warp-uniform
        const uint4 *src = reinterpret_cast<const uint4 *>(raw + s * kRawStageBytes + r * (kDI / 2));
        uint4 in[kDI / 32];
#pragma unroll
        for (int q = 0; q < kDI / 32; ++q) in[q] = src[q];
        uint8_t *dst = stage + sc2 * kStageBytes + r * kDI;
#pragma unroll
        for (int q = 0; q < kDI / 32; ++q) {   // 32 codes -> two 16-byte chunks
          uint32_t o[8];
          e2m1x8_to_e4m3x8(in[q].x, o[0], o[1]);
          e2m1x8_to_e4m3x8(in[q].y, o[2], o[3]);
          e2m1x8_to_e4m3x8(in[q].z, o[4], o[5]);
          e2m1x8_to_e4m3x8(in[q].w, o[6], o[7]);
          *reinterpret_cast<uint4 *>(dst + (((2 * q) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4 *>(dst + (((2 * q + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor-core reads
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&empty[s]);     // raw stage free for the next copy
          mbar_arrive(&cfull[sc2]);   // converted tile ready
        }
      }
    }
    for (int it0 = grp; it0 < n_it && live; it0 += 4 * n_grp) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = it0 + n_grp * u;
        if (it >= n_it || !live) break;
        const int acc = it % n_acc;
        const uint32_t aph = (uint32_t)(it / n_acc) & 1u;
        const bool ok = mbar_wait(&tfull[acc], aph, abort_flag, a.status, a.wait_limit);
        if (!__all_sync(0xffffffffu, ok)) { live = false; break; }   // warp-uniform: TMEM loads are .sync.aligned
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(g * 32) << 16) + (uint32_t)(acc * 2 * H);
        float s4[4] = {0.f, 0.f, 0.f, 0.f};   // independent partial sums (no 64-deep FMA chain)
        for (int c0 = 0; c0 < H; c0 += 32) {
          uint32_t hv[32], lv[32];
          tmem_ld32(taddr + c0, hv);
          if (a.hi_only) {
#pragma unroll
            for (int q = 0; q < 32; ++q) lv[q] = 0u;
          } else {
            tmem_ld32(taddr + H + c0, lv);
          }
          tmem_wait_ld();
          // w_h/S_h as 16-byte shared loads: a quarter of the shared-memory wavefronts of
          // scalar loads (shared-memory bandwidth is shared with the TMA writes and MMA reads)
          const float4 *wq4 = reinterpret_cast<const float4 *>(wq + c0);
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {
            const float4 wv = wq4[h4];
            const float wk[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int h = 4 * h4 + e;
              s4[e] = fmaf(wk[e], fmaxf(fmaf(__uint_as_float(lv[h]), 0.0625f, __uint_as_float(hv[h])), 0.f), s4[e]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        const float sum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        const long long j = (tile_lo + it) * kTileM + g * 32 + lane;
        if (j < n_vis) {
          const float v = sum * sc[u];
          a.scores[(long long)row * a.stride + j] = v;
          if (a.hist) atomicAdd(&shist[float_key(v) >> (32 - kPrefixBits)], 1u);
        }
        sc[u] = scale_of(it + 4 * n_grp, pgn[u]);
        pgn[u] = page_of(it + 8 * n_grp);
      }
    }
  }
  // Warps 0 and 1 ran their loops on lane 0 only: reconverge each warp before the
  // CTA barrier, which counts warps (a warp arriving in two parts would be counted
  // twice and release the barrier while epilogue warps still read TMEM).
  __syncwarp();
  __syncthreads();
  if (*abort_flag) {   // uniform: a wait gave up.  Nothing may be in flight when the CTA leaves:
    if (warp == 0 && lane == 0) {   // the key copies already issued land in shared memory,
      for (int it = issued > kStages ? issued - kStages : 0; it < issued; ++it)
        for (int i = 0; i < (1 << 20) && !mbar_try_wait(&full[it % kStages], (uint32_t)(it / kStages) & 1u); ++i) {
        }
    }
    if (warp == 1 && lane == 0) {   // and the MMAs already issued finish before TMEM is freed
      umma_commit(drain);
      for (int i = 0; i < (1 << 20) && !mbar_try_wait(drain, 0u); ++i) {
      }
    }
    __syncthreads();
  }
  if (a.hist) {   // this CTA's prefix counts into the row's histogram
    for (int e = threadIdx.x; e < kPrefixBins; e += kThreads) {
      const unsigned v = shist[e];
      if (v) atomicAdd(a.hist + (long long)row * kPrefixBins + e, v);
    }
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

bool index_tc_supported(const CacheView &c, int heads_idx) {
  if (c.kv_dtype != CSA_E4M3 || c.d_idx != kDI) return false;
  if (heads_idx != 32 && heads_idx != 64 && heads_idx != 128) return false;
  if (c.page_size != 0) {
    const int p = c.page_size;
    if (p < 8 || (p & (p - 1))) return false;
  }
  return true;
}

size_t index_tc_smem_bytes() {
  return 1024 + (size_t)kStages * kStageBytes + 2 * 128 * kDI + 128 * sizeof(float) + (2 * kStages + 8 + 2 * kConvStages) * 8 + 16 +
         (size_t)kPrefixBins * sizeof(unsigned);
}

cudaError_t launch_index_tc(const CacheView &c, int batch, int n_q, const void *q_idx, int q_dtype, const float *w,
                            int heads_idx, float *scores, long long stride, int num_sms, int *status,
                            const TopkArea *area, const IndexDebug &dbg, cudaStream_t st) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap map;
  const int box_rows = c.page_size == 0 ? kTileM : (c.page_size < kTileM ? c.page_size : kTileM);
  // contiguous: the real row extent, so a tail tile past it reads zeros; paged:
  // rows are reached only through valid page ids, the extent is not known here
  const cuuint64_t rows = c.page_size == 0 ? (cuuint64_t)batch * (cuuint64_t)c.max_entries : (cuuint64_t)0x7fffffff;
  // e4m3 keys: 128-byte rows, 128-byte swizzle (the MMA reads the tile in place);
  // FP4 keys: 64-byte packed rows, unswizzled (the converter reads them row by row)
  const cuuint64_t row_bytes = c.idx_fp4 ? kDI / 2 : kDI;
  cuuint64_t gdim[2] = {row_bytes, rows};
  cuuint64_t gstride[1] = {row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)row_bytes, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, (void *)c.idx_key, gdim, gstride, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, c.idx_fp4 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  TcArgs a;
  a.c = c; a.n_q = n_q; a.heads = heads_idx; a.q_dtype = q_dtype;
  a.q_idx = (const uint8_t *)q_idx; a.w = w; a.scores = scores; a.stride = stride;
  a.box_rows = box_rows; a.status = status;
  a.wait_limit = dbg.wait_limit > 0 ? dbg.wait_limit : (1LL << 24);
  a.starve = dbg.starve;
  a.q_vec = ((uintptr_t)q_idx & 15) == 0;
  a.hi_only = q_dtype == CSA_BF16_Q_E4M3;
  a.fp4 = c.idx_fp4;
  if (a.hi_only) a.q_dtype = CSA_BF16;   // the input is bf16 either way
  a.hist = area ? area->hist : nullptr;
  a.sel_ctr = area ? area->ctr : nullptr;
  a.sel_ctr_words = area && area->ctr ? area->rows * (4 + kDigitBins) : 0;
  const int rows_q = batch * n_q;
  a.rows = rows_q;
  a.grid_sms = num_sms;
  dim3 grid;
  if (rows_q >= num_sms || rows_q > kMaxFlatRows) {   // a row per CTA
    a.ctas_per_row = 1;
    grid = dim3(1, rows_q);
  } else {                   // flat grid, CTAs split over rows by their tile counts
    a.ctas_per_row = 0;       // (ceil(tiles / L) per row, <= SMs in all)
    grid = dim3(num_sms, 1);
  }
  const size_t smem = index_tc_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(k_index_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_index_tc, grid, dim3(kThreads), smem, st, 1, map, a);
}

}  // namespace csa
