// Host side of the C ABI declared in include/csa.h: argument checks, workspace
// layout, rotary phase tables and kernel launches.  No device memory is
// allocated here; every buffer comes from the caller.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

#include "kernels.h"

namespace {

thread_local std::string g_err;

// Failure-injection settings of the indexer's bounded waits (csa_debug_set); read at
// every launch.
std::atomic<long long> g_wait_limit{0};
std::atomic<int> g_starve{0};

csa_status fail(csa_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

csa_status ok() {
  g_err.clear();
  return CSA_OK;
}

csa_status cuda_status(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return ok();
  return fail(CSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool a16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

long long entry_cap(const csa_cache *c) {
  return c->page_size ? (long long)c->max_pages * c->page_size : (long long)c->max_entries;
}

csa_status check_cache(const csa_cache *c) {
  if (!c) return fail(CSA_ERR_INVALID_ARG, "cache is NULL");
  if (c->m < 1 || c->m > 1024) return fail(CSA_ERR_INVALID_ARG, "m=%d outside [1,1024]", c->m);
  if (c->d_rope < 0 || c->d_rope > 64 || c->d_rope % 8 || c->d_rope > c->d)
    return fail(CSA_ERR_INVALID_ARG, "d_rope=%d must be a multiple of 8 in [0,min(64,d)]", c->d_rope);
  if (c->d < 16 || c->d % 16 || (c->d - c->d_rope) % 16)
    return fail(CSA_ERR_INVALID_ARG, "d=%d: d and d-d_rope must be multiples of 16", c->d);
  if (!(c->d_idx == 0 || c->d_idx == 16 || c->d_idx == 32 || c->d_idx == 64 || c->d_idx == 128))
    return fail(CSA_ERR_UNSUPPORTED, "d_idx=%d not in {0,16,32,64,128}", c->d_idx);
  if (c->d + c->d_idx > 1024) return fail(CSA_ERR_UNSUPPORTED, "d + d_idx = %d > 1024", c->d + c->d_idx);
  if (c->kv_dtype != CSA_E4M3 && c->kv_dtype != CSA_F32)
    return fail(CSA_ERR_INVALID_ARG, "kv_dtype must be CSA_E4M3 or CSA_F32");
  if (c->win_dtype != CSA_BF16 && c->win_dtype != CSA_F32)
    return fail(CSA_ERR_INVALID_ARG, "win_dtype must be CSA_BF16 or CSA_F32");
  if (c->n_win < 1) return fail(CSA_ERR_INVALID_ARG, "n_win must be >= 1");
  if (c->win_cap < c->n_win) return fail(CSA_ERR_INVALID_ARG, "win_cap=%d < n_win=%d", c->win_cap, c->n_win);
  if (!(c->rope_theta > 1.0)) return fail(CSA_ERR_INVALID_ARG, "rope_theta must be > 1");
  if (c->page_size < 0) return fail(CSA_ERR_INVALID_ARG, "page_size < 0");
  if (c->page_size > 0) {
    if (!c->page_table || c->max_pages < 1) return fail(CSA_ERR_INVALID_ARG, "paged cache needs page_table, max_pages");
  } else if (c->max_entries < 1) {
    return fail(CSA_ERR_INVALID_ARG, "max_entries must be >= 1");
  }
  if (!c->kv_nope || !c->kv_rope || !c->win || !c->pool_state || !c->n_tokens)
    return fail(CSA_ERR_INVALID_ARG, "cache pointer is NULL");
  if (c->kv_dtype == CSA_E4M3 && !c->kv_scale) return fail(CSA_ERR_INVALID_ARG, "kv_scale is NULL");
  if (c->d_idx > 0 && (!c->idx_key || (c->kv_dtype == CSA_E4M3 && !c->idx_scale)))
    return fail(CSA_ERR_INVALID_ARG, "indexer key pointers are NULL");
  if (c->idx_dtype != 0 && c->idx_dtype != CSA_E2M1)
    return fail(CSA_ERR_INVALID_ARG, "idx_dtype must be 0 (as kv_dtype) or CSA_E2M1");
  if (c->idx_dtype == CSA_E2M1 && (c->kv_dtype != CSA_E4M3 || c->d_idx < 32))
    return fail(CSA_ERR_UNSUPPORTED, "FP4 indexer keys need kv_dtype E4M3 and d_idx in {32, 64, 128}");
  if (!a16(c->kv_nope) || !a16(c->kv_rope) || !a16(c->win) || !a16(c->pool_state) || !a16(c->idx_key) ||
      ((uintptr_t)c->kv_scale & 3) || ((uintptr_t)c->idx_scale & 3) || ((uintptr_t)c->n_tokens & 7))
    return fail(CSA_ERR_INVALID_ARG, "cache arrays must be 16-byte aligned");
  return ok();
}

csa::CacheView view(const csa_cache *c) {
  csa::CacheView v;
  v.m = c->m; v.d = c->d; v.d_rope = c->d_rope; v.d_idx = c->d_idx; v.kv_dtype = c->kv_dtype;
  v.win_dtype = c->win_dtype; v.n_win = c->n_win; v.win_cap = c->win_cap; v.page_size = c->page_size;
  v.max_pages = c->max_pages; v.max_entries = c->max_entries; v.cap = entry_cap(c);
  v.kv_nope = (const uint8_t *)c->kv_nope; v.kv_scale = c->kv_scale; v.kv_rope = (const uint8_t *)c->kv_rope;
  v.idx_key = (const uint8_t *)c->idx_key; v.idx_scale = c->idx_scale; v.page_table = c->page_table;
  v.win = (const uint8_t *)c->win; v.pool_state = c->pool_state; v.n_tokens = (long long *)c->n_tokens;
  v.idx_fp4 = c->idx_dtype == CSA_E2M1;
  return v;
}

// Fixed-point phase increment per rotary frequency: round(2^64 * f_i / (2 pi)),
// f_i = theta^(-2i/d_rope), evaluated in x87 extended precision.
csa::RopeTable rope_table(double theta, int d_rope) {
  thread_local double last_theta = -1;
  thread_local int last_dr = -1;
  thread_local csa::RopeTable tab;
  if (theta == last_theta && d_rope == last_dr) return tab;
  std::memset(&tab, 0, sizeof(tab));
  const long double two_pi = 6.283185307179586476925286766559005768L;
  for (int i = 0; i < d_rope / 2; ++i) {
    const long double f = powl((long double)theta, -2.0L * i / (long double)d_rope);
    const long double turns = f / two_pi;                       // in (0, 1)
    tab.step[i] = (unsigned long long)llroundl(ldexpl(turns, 64));   // < 2^62
  }
  last_theta = theta;
  last_dr = d_rope;
  return tab;
}

int num_sms() {
  thread_local int dev = -1, n = 148;
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return n;
  if (cur != dev) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, cur) == cudaSuccess && v > 0) n = v;
    dev = cur;
  }
  return n;
}

constexpr size_t kHeader = 256;
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct AttendPlan {
  bool tc;
  int n_splits, cps;
  size_t part_o_bytes, part_ml_bytes;
};

// one_split: the prefill plan (one CTA walks all of a row's chunks) whatever n_q is;
// dense: the key list is every visible entry (no top-k list)
AttendPlan attend_plan(const csa_cache *c, int batch, int n_q, int heads, long long list_cap, bool one_split = false,
                       bool dense = false) {
  AttendPlan p;
  p.tc = csa::attend_tc_supported(view(c), heads, CSA_BF16);
  csa::attend_plan(one_split ? 2 : n_q, list_cap, c->n_win, p.tc, dense && c->d >= 256, p.n_splits, p.cps);
  const size_t parts = (size_t)batch * n_q * p.n_splits * heads;
  p.part_o_bytes = p.n_splits > 1 ? align256(parts * c->d * sizeof(float)) : 0;
  p.part_ml_bytes = p.n_splits > 1 ? align256(parts * 2 * sizeof(float)) : 0;
  return p;
}

size_t scores_bytes(const csa_cache *c, int batch, int n_q) {
  return align256((size_t)batch * n_q * entry_cap(c) * sizeof(float));
}

// The top-k area of a fused index + top-k call (decode-sized calls only: prefix
// histograms and the row-split top-k's counters, slots and lists) sits at the end of
// the workspace, 256-byte aligned, clear of the scores and of the attention's split
// partials (both start after the header); csa_workspace_size reserves it.  0 bytes
// when the call has too many rows for it.
size_t area_bytes(const csa_cache *c, int batch, int n_q, int k) {
  const long long rows = (long long)batch * n_q;
  return rows <= csa::kPrefixRowsMax ? csa::topk_area_bytes((int)rows, entry_cap(c), k) : 0;
}

csa_status check_ws(void *ws, size_t ws_bytes, size_t need) {
  if (need == 0) return ok();
  if (!ws) return fail(CSA_ERR_WORKSPACE, "workspace is NULL (need %zu bytes)", need);
  if (((uintptr_t)ws & 255u)) return fail(CSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < need) return fail(CSA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  return ok();
}

csa_status check_q(int batch, int n_q, const csa_cache *c) {
  if (batch < 1 || n_q < 1) return fail(CSA_ERR_INVALID_ARG, "batch=%d n_q=%d must be >= 1", batch, n_q);
  if ((long long)c->win_cap < (long long)c->n_win + n_q - 1)
    return fail(CSA_ERR_INVALID_ARG, "win_cap=%d < n_win + n_q - 1 = %d", c->win_cap, c->n_win + n_q - 1);
  return ok();
}

// no_entries: a sliding-window-only layer -- the key list is the window alone (the
// cache view's entry capacity is 0, so no entry is ever visible or read)
csa_status attend_common(const csa_cache *c, int batch, int n_q, const void *q, int q_dtype, int heads,
                         const float *sink, const int32_t *idx, int k, void *out, int out_dtype, float *out_lse,
                         void *ws, size_t ws_bytes, cudaStream_t st, bool no_entries = false,
                         bool one_split = false) {
  csa_status s = check_cache(c);
  if (s) return s;
  if ((s = check_q(batch, n_q, c))) return s;
  if (heads < 1 || heads > 128) return fail(CSA_ERR_UNSUPPORTED, "heads=%d outside [1,128]", heads);
  if (!q || !sink || !out) return fail(CSA_ERR_INVALID_ARG, "q, sink and out must be non-NULL");
  if (q_dtype != CSA_BF16 && q_dtype != CSA_F32) return fail(CSA_ERR_INVALID_ARG, "q_dtype must be BF16 or F32");
  if (out_dtype != CSA_BF16 && out_dtype != CSA_F32) return fail(CSA_ERR_INVALID_ARG, "out_dtype must be BF16 or F32");
  if (idx && k < 1) return fail(CSA_ERR_INVALID_ARG, "k must be >= 1");
  if (((uintptr_t)q & 15) || ((uintptr_t)out & 7) || ((uintptr_t)idx & 3) || ((uintptr_t)out_lse & 3))
    return fail(CSA_ERR_INVALID_ARG, "q must be 16-byte, out 8-byte, idx and out_lse 4-byte aligned");
  if (csa::attend_smem_bytes(c->d) > 227 * 1024) return fail(CSA_ERR_UNSUPPORTED, "d=%d too large", c->d);
  const long long list_cap = no_entries ? 0 : idx ? (long long)k : entry_cap(c);
  const AttendPlan p = attend_plan(c, batch, n_q, heads, list_cap, one_split, !no_entries && !idx);
  const size_t need = p.n_splits > 1 ? kHeader + p.part_o_bytes + p.part_ml_bytes : 0;
  if ((s = check_ws(ws, ws_bytes, need))) return s;
  csa::AttendArgs a;
  a.c = view(c);
  if (no_entries) a.c.cap = 0;
  a.rope = rope_table(c->rope_theta, c->d_rope);
  a.n_q = n_q; a.heads = heads; a.q_dtype = q_dtype; a.out_dtype = out_dtype;
  a.q = (const uint8_t *)q; a.sink = sink; a.idx = idx; a.k = k;
  a.n_splits = p.n_splits; a.chunks_per_split = p.cps;
  a.keys_per_split = p.cps * (p.tc ? 64 : csa::kKC);
  a.part_o = need ? (float *)((char *)ws + kHeader) : nullptr;
  a.part_ml = need ? (float *)((char *)ws + kHeader + p.part_o_bytes) : nullptr;
  a.out = (uint8_t *)out; a.out_lse = out_lse;
  a.scale = (float)(1.0 / std::sqrt((double)c->d));
  return cuda_status(p.tc ? csa::launch_attend_tc(a, batch * n_q, st) : csa::launch_attend(a, batch * n_q, st),
                     "attention launch");
}

csa_status check_index_args(const csa_cache *c, int batch, int n_q, const void *q_idx, int q_dtype, const float *w,
                            int heads_idx) {
  csa_status s = check_cache(c);
  if (s) return s;
  if ((s = check_q(batch, n_q, c))) return s;
  if (c->d_idx == 0) return fail(CSA_ERR_INVALID_ARG, "cache has no indexer stream (d_idx == 0)");
  if (heads_idx < 1 || heads_idx > 128) return fail(CSA_ERR_UNSUPPORTED, "heads_idx=%d outside [1,128]", heads_idx);
  if (!q_idx || !w) return fail(CSA_ERR_INVALID_ARG, "q_idx and w must be non-NULL");
  if (q_dtype != CSA_BF16 && q_dtype != CSA_F32 && q_dtype != CSA_BF16_Q_E4M3)
    return fail(CSA_ERR_INVALID_ARG, "q_dtype must be BF16, F32 or BF16_Q_E4M3");
  if ((size_t)heads_idx * (c->d_idx + 1) * sizeof(float) > 227 * 1024)
    return fail(CSA_ERR_UNSUPPORTED, "indexer query too large");
  return ok();
}

// Indexer dispatch: the tensor-core kernel for e4m3 keys of dim 128 and 32/64/128
// heads; the CUDA-core kernel otherwise (fp32 caches, other dims).
// area (may be null): the top-k area, whose prefix histograms only the tensor-core
// indexer fills (and whose row counters it zeroes); *hist_used tells the caller
// whether it did
cudaError_t launch_indexer(const csa_cache *c, int batch, int n_q, const void *q_idx, int q_dtype, const float *w,
                           int heads_idx, float *scores, long long stride, void *ws, cudaStream_t st,
                           const csa::TopkArea *area = nullptr, bool *hist_used = nullptr) {
  const csa::CacheView v = view(c);
  if (hist_used) *hist_used = false;
  if (csa::index_tc_supported(v, heads_idx)) {
    if (hist_used) *hist_used = area != nullptr;
    const csa::IndexDebug dbg{g_wait_limit.load(), g_starve.load()};
    return csa::launch_index_tc(v, batch, n_q, q_idx, q_dtype, w, heads_idx, scores, stride, num_sms(),
                                ws ? (int *)ws : nullptr, area, dbg, st);
  }
  return csa::launch_index_generic(v, batch, n_q, q_idx, q_dtype, w, heads_idx, scores, stride, entry_cap(c), st);
}

}  // namespace

namespace {

// A sliding-window-only layer's cache as the attention path sees it: the window ring
// and the token counts; m, the entry storage and the indexer stream are ignored (the
// entry fields get stand-ins that are never read: the entry capacity is 0).
csa_status swa_view(const csa_cache *c, csa_cache &cc) {
  if (!c) return fail(CSA_ERR_INVALID_ARG, "cache is NULL");
  if (!c->win || !c->n_tokens) return fail(CSA_ERR_INVALID_ARG, "win and n_tokens must be non-NULL");
  cc = *c;
  cc.m = 1; cc.d_idx = 0; cc.page_size = 0; cc.max_pages = 0; cc.max_entries = 1;
  cc.kv_dtype = c->win_dtype == CSA_BF16 ? CSA_E4M3 : CSA_F32;
  cc.kv_nope = c->win; cc.kv_rope = c->win; cc.kv_scale = reinterpret_cast<float *>(c->win);
  cc.idx_key = nullptr; cc.idx_scale = nullptr; cc.page_table = nullptr;
  cc.pool_state = reinterpret_cast<float *>(c->win);
  return check_cache(&cc);
}

// Sequence b of a cache as a cache of one sequence (pointer offsets only).
csa_cache seq_view(const csa_cache *c, int b) {
  csa_cache s = *c;
  const size_t eb = c->kv_dtype == CSA_E4M3 ? 1 : 4;   // bytes per non-rotary / indexer-key element
  if (c->page_size == 0) {
    const size_t r0 = (size_t)b * (size_t)c->max_entries;
    s.kv_nope = (uint8_t *)c->kv_nope + r0 * (c->d - c->d_rope) * eb;
    s.kv_rope = (uint8_t *)c->kv_rope + r0 * c->d_rope * (c->kv_dtype == CSA_E4M3 ? 2 : 4);
    if (c->kv_scale) s.kv_scale = c->kv_scale + r0;
    if (c->idx_key) s.idx_key = (uint8_t *)c->idx_key + r0 * (c->idx_dtype == CSA_E2M1 ? c->d_idx / 2 : c->d_idx * eb);
    if (c->idx_scale) s.idx_scale = c->idx_scale + r0;
  } else {
    s.page_table = c->page_table + (size_t)b * c->max_pages;
  }
  s.win = (uint8_t *)c->win + (size_t)b * c->win_cap * c->d * (c->win_dtype == CSA_F32 ? 4 : 2);
  s.pool_state = c->pool_state + (size_t)b * 3 * (c->d + c->d_idx);
  s.n_tokens = c->n_tokens + b;
  return s;
}

}  // namespace

// Scratch of csa_index_topk_static: one array per device, reused by every call.
static __device__ __align__(256) unsigned char g_static_scratch[CSA_STATIC_SCRATCH_BYTES];

namespace {

// Device address of g_static_scratch on the current device, looked up once per
// device (cudaGetSymbolAddress with that device current).  Host code only sees
// a host-side stand-in for the array; kernels must get this address instead.
void *static_scratch(csa_status &st) {
  static std::mutex mu;
  static void *addr[256] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 256) {
    st = cuda_status(e == cudaSuccess ? cudaErrorInvalidDevice : e, "current device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p) {
      st = cuda_status(e == cudaSuccess ? cudaErrorInvalidSymbol : e, "static scratch address");
      return nullptr;
    }
    addr[dev] = p;
  }
  st = CSA_OK;
  return addr[dev];
}

}  // namespace

extern "C" {

int csa_version(void) { return 100; }

const char *csa_last_error(void) { return g_err.c_str(); }

size_t csa_workspace_size(const csa_cache *c, int batch, int n_q, int heads, int k) {
  if (check_cache(c) || batch < 1 || n_q < 1 || heads < 1) return 0;
  size_t need = kHeader;
  if (k > 0) need = std::max(need, kHeader + scores_bytes(c, batch, n_q));
  const AttendPlan p = attend_plan(c, batch, n_q, heads, k > 0 ? (long long)k : entry_cap(c), false, k <= 0);
  need = std::max(need, kHeader + p.part_o_bytes + p.part_ml_bytes);
  if (k > 0) need = ((need + 255) & ~(size_t)255) + area_bytes(c, batch, n_q, k);
  return need;
}

csa_status csa_compress(const csa_cache *c, int batch, int n_new, const void *x, const void *gate, const void *idx_x,
                        const void *idx_gate, const float *pos_bias, const float *idx_pos_bias, int in_dtype,
                        csa_stream_t stream) {
  csa_status s = check_cache(c);
  if (s) return s;
  if (batch < 1 || n_new < 1) return fail(CSA_ERR_INVALID_ARG, "batch=%d n_new=%d must be >= 1", batch, n_new);
  if (in_dtype != c->win_dtype) return fail(CSA_ERR_INVALID_ARG, "in_dtype must equal the ring dtype");
  if (!x || !gate || !pos_bias) return fail(CSA_ERR_INVALID_ARG, "x, gate and pos_bias must be non-NULL");
  if (c->d_idx > 0 && (!idx_x || !idx_gate || !idx_pos_bias))
    return fail(CSA_ERR_INVALID_ARG, "indexer-key inputs must be non-NULL when d_idx > 0");
  return cuda_status(csa::launch_compress(view(c), rope_table(c->rope_theta, c->d_rope), batch, n_new, in_dtype, x,
                                          gate, idx_x, idx_gate, pos_bias, idx_pos_bias, (cudaStream_t)stream),
                     "compress launch");
}

csa_status csa_index_scores(const csa_cache *c, int batch, int n_q, const void *q_idx, int q_dtype, const float *w,
                            int heads_idx, float *scores, int64_t stride, void *ws, size_t ws_bytes,
                            csa_stream_t stream) {
  csa_status s = check_index_args(c, batch, n_q, q_idx, q_dtype, w, heads_idx);
  if (s) return s;
  if (!scores) return fail(CSA_ERR_INVALID_ARG, "scores is NULL");
  if (stride < entry_cap(c)) return fail(CSA_ERR_INVALID_ARG, "scores_stride %lld < entry capacity %lld",
                                         (long long)stride, entry_cap(c));
  if (ws && ((uintptr_t)ws & 255u)) return fail(CSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws && ws_bytes < kHeader) return fail(CSA_ERR_WORKSPACE, "workspace smaller than its %zu-byte header", kHeader);
  return cuda_status(launch_indexer(c, batch, n_q, q_idx, q_dtype, w, heads_idx, scores, stride, ws,
                                    (cudaStream_t)stream),
                     "indexer launch");
}

csa_status csa_topk(const csa_cache *c, int batch, int n_q, const float *scores, int64_t stride, int k,
                    int32_t *out_idx, int32_t *out_count, void *ws, size_t ws_bytes, csa_stream_t stream) {
  csa_status s = check_cache(c);
  if (s) return s;
  if (batch < 1 || n_q < 1) return fail(CSA_ERR_INVALID_ARG, "batch and n_q must be >= 1");
  if (k < 1) return fail(CSA_ERR_INVALID_ARG, "k must be >= 1");
  if (!scores || !out_idx || !out_count) return fail(CSA_ERR_INVALID_ARG, "NULL pointer");
  if (stride < 1) return fail(CSA_ERR_INVALID_ARG, "scores_stride must be >= 1");
  if (ws && ((uintptr_t)ws & 255u)) return fail(CSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  // the workspace's status word (a failed indexer call on it): rows report count -1
  const int *status = ws && ws_bytes >= kHeader ? (const int *)ws : nullptr;
  return cuda_status(csa::launch_topk(view(c), batch, n_q, scores, stride, k, out_idx, out_count, nullptr, num_sms(),
                                      status, (cudaStream_t)stream),
                     "top-k launch");
}

csa_status csa_index_topk(const csa_cache *c, int batch, int n_q, const void *q_idx, int q_dtype, const float *w,
                          int heads_idx, int k, int32_t *out_idx, int32_t *out_count, void *ws, size_t ws_bytes,
                          csa_stream_t stream) {
  csa_status s = check_index_args(c, batch, n_q, q_idx, q_dtype, w, heads_idx);
  if (s) return s;
  if (k < 1) return fail(CSA_ERR_INVALID_ARG, "k must be >= 1");
  if (!out_idx || !out_count) return fail(CSA_ERR_INVALID_ARG, "NULL output pointer");
  const size_t need = kHeader + scores_bytes(c, batch, n_q);
  if ((s = check_ws(ws, ws_bytes, need))) return s;
  float *scores = (float *)((char *)ws + kHeader);
  const long long cap = entry_cap(c);
  // the top-k area when the workspace has room for it (sized by csa_workspace_size)
  const size_t hb = area_bytes(c, batch, n_q, k);
  const size_t ho = ws_bytes >= hb ? (ws_bytes - hb) & ~(size_t)255 : 0;
  csa::TopkArea area;
  const bool has_area = hb && ho >= need;
  if (has_area) area = csa::topk_area((char *)ws + ho, batch * n_q, cap, k);
  bool used = false;
  cudaError_t e = launch_indexer(c, batch, n_q, q_idx, q_dtype, w, heads_idx, scores, cap, ws, (cudaStream_t)stream,
                                 has_area ? &area : nullptr, &used);
  if (e != cudaSuccess) return cuda_status(e, "indexer launch");
  return cuda_status(csa::launch_topk(view(c), batch, n_q, scores, cap, k, out_idx, out_count, used ? &area : nullptr,
                                      num_sms(), (const int *)ws, (cudaStream_t)stream),
                     "top-k launch");
}

csa_status csa_index_topk_static(const csa_cache *c, int batch, int n_q, const void *q_idx, int q_dtype,
                                 const float *w, int heads_idx, int k, int32_t *out_idx, int32_t *out_count,
                                 csa_stream_t stream) {
  csa_status s = check_index_args(c, batch, n_q, q_idx, q_dtype, w, heads_idx);
  if (s) return s;
  if (k < 1) return fail(CSA_ERR_INVALID_ARG, "k must be >= 1");
  if (!out_idx || !out_count) return fail(CSA_ERR_INVALID_ARG, "NULL output pointer");
  const size_t need = kHeader + scores_bytes(c, batch, n_q);
  if (need > CSA_STATIC_SCRATCH_BYTES)
    return fail(CSA_ERR_WORKSPACE,
                "needs %zu bytes of scratch (%d rows x %lld entries); the static scratch holds %zu bytes",
                need, batch * n_q, entry_cap(c), (size_t)CSA_STATIC_SCRATCH_BYTES);
  void *ws = static_scratch(s);
  if (!ws) return s;
  cudaError_t e = cudaMemsetAsync(ws, 0, kHeader, (cudaStream_t)stream);   // status word starts at zero
  if (e != cudaSuccess) return cuda_status(e, "static scratch clear");
  float *scores = (float *)((char *)ws + kHeader);
  const long long cap = entry_cap(c);
  e = launch_indexer(c, batch, n_q, q_idx, q_dtype, w, heads_idx, scores, cap, ws, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e, "indexer launch");
  return cuda_status(csa::launch_topk(view(c), batch, n_q, scores, cap, k, out_idx, out_count, nullptr, num_sms(),
                                      (const int *)ws, (cudaStream_t)stream),
                     "top-k launch");
}

csa_status csa_sparse_attend(const csa_cache *c, int batch, int n_q, const void *q, int q_dtype, int heads,
                             const float *sink, const int32_t *idx, int k, void *out, int out_dtype, float *out_lse,
                             void *ws, size_t ws_bytes, csa_stream_t stream) {
  if (!idx) return fail(CSA_ERR_INVALID_ARG, "idx is NULL");
  return attend_common(c, batch, n_q, q, q_dtype, heads, sink, idx, k, out, out_dtype, out_lse, ws, ws_bytes,
                       (cudaStream_t)stream);
}

csa_status hca_attend(const csa_cache *c, int batch, int n_q, const void *q, int q_dtype, int heads,
                      const float *sink, void *out, int out_dtype, float *out_lse, void *ws, size_t ws_bytes,
                      csa_stream_t stream) {
  return attend_common(c, batch, n_q, q, q_dtype, heads, sink, nullptr, 0, out, out_dtype, out_lse, ws, ws_bytes,
                       (cudaStream_t)stream);
}

size_t swa_workspace_size(const csa_cache *c, int batch, int n_q, int heads) {
  csa_cache cc;
  if (swa_view(c, cc) || batch < 1 || n_q < 1 || heads < 1) return 0;
  const AttendPlan p = attend_plan(&cc, batch, n_q, heads, 0);
  return kHeader + p.part_o_bytes + p.part_ml_bytes;
}

csa_status swa_append(const csa_cache *c, int batch, int n_new, const void *x, int in_dtype, csa_stream_t stream) {
  csa_cache cc;
  csa_status s = swa_view(c, cc);
  if (s) return s;
  if (batch < 1 || n_new < 1) return fail(CSA_ERR_INVALID_ARG, "batch=%d n_new=%d must be >= 1", batch, n_new);
  if (in_dtype != c->win_dtype) return fail(CSA_ERR_INVALID_ARG, "in_dtype must equal the ring dtype");
  if (!x || ((uintptr_t)x & 15)) return fail(CSA_ERR_INVALID_ARG, "x must be non-NULL and 16-byte aligned");
  return cuda_status(csa::launch_swa_append(view(&cc), batch, n_new, in_dtype, x, (cudaStream_t)stream),
                     "window append launch");
}

csa_status swa_attend(const csa_cache *c, int batch, int n_q, const void *q, int q_dtype, int heads, const float *sink,
                      void *out, int out_dtype, float *out_lse, void *ws, size_t ws_bytes, csa_stream_t stream) {
  csa_cache cc;
  csa_status s = swa_view(c, cc);
  if (s) return s;
  return attend_common(&cc, batch, n_q, q, q_dtype, heads, sink, nullptr, 0, out, out_dtype, out_lse, ws, ws_bytes,
                       (cudaStream_t)stream, true);
}

// Workspace of the calls one chunk of at most `chunk` rows makes: the largest over the
// chunk lengths a call can see (the prefix histograms are reserved only for calls of
// at most kPrefixRowsMax rows, so the size is not monotone in the rows).
static size_t prefill_inner(const csa_cache *c, int chunk, int heads, int k) {
  const csa_cache s = seq_view(c, 0);
  const size_t a = csa_workspace_size(&s, 1, chunk, heads, k);
  const size_t b = csa_workspace_size(&s, 1, std::min(chunk, csa::kPrefixRowsMax), heads, k);
  return (a == 0 || b == 0) ? 0 : align256(std::max(a, b));
}

size_t csa_prefill_workspace_size(const csa_cache *c, int chunk, int heads, int k) {
  if (check_cache(c) || chunk < 1 || heads < 1 || k < 1) return 0;
  const size_t inner = prefill_inner(c, chunk, heads, k);
  if (inner == 0) return 0;
  return inner + align256((size_t)chunk * k * sizeof(int32_t)) + align256((size_t)chunk * sizeof(int32_t));
}

csa_status csa_prefill_chunked(const csa_cache *c, int batch, int n_new, int chunk, const void *x, const void *gate,
                               const void *idx_x, const void *idx_gate, const float *pos_bias,
                               const float *idx_pos_bias, int in_dtype, const void *q_idx, int q_idx_dtype,
                               const float *w, int heads_idx, const void *q, int q_dtype, int heads,
                               const float *sink, int k, void *out, int out_dtype, float *out_lse, void *ws,
                               size_t ws_bytes, csa_stream_t stream) {
  csa_status s = check_cache(c);
  if (s) return s;
  if (batch < 1 || n_new < 1 || chunk < 1) return fail(CSA_ERR_INVALID_ARG, "batch, n_new and chunk must be >= 1");
  if (c->d_idx == 0) return fail(CSA_ERR_INVALID_ARG, "cache has no indexer stream (d_idx == 0)");
  if (!x || !gate || !idx_x || !idx_gate || !q_idx || !w || !q || !sink || !out)
    return fail(CSA_ERR_INVALID_ARG, "NULL input or output pointer");
  const size_t need = csa_prefill_workspace_size(c, std::min(chunk, n_new), heads, k);
  if (need == 0) return fail(CSA_ERR_INVALID_ARG, "invalid prefill geometry");
  if ((s = check_ws(ws, ws_bytes, need))) return s;
  const int L0 = std::min(chunk, n_new);
  const size_t inner = prefill_inner(c, L0, heads, k);
  int32_t *idx = (int32_t *)((char *)ws + inner);
  int32_t *cnt = (int32_t *)((char *)ws + inner + align256((size_t)L0 * k * sizeof(int32_t)));
  const size_t tb = in_dtype == CSA_F32 ? 4 : 2, qb = q_dtype == CSA_F32 ? 4 : 2;
  const size_t qib = q_idx_dtype == CSA_F32 ? 4 : 2, ob = out_dtype == CSA_F32 ? 4 : 2;
  for (int b = 0; b < batch; ++b) {
    const csa_cache sc = seq_view(c, b);
    for (int p0 = 0; p0 < n_new; p0 += chunk) {
      const int L = std::min(chunk, n_new - p0);
      const size_t r0 = (size_t)b * n_new + p0;   // first row of this chunk in the [batch][n_new] inputs
      const size_t inner_l = csa_workspace_size(&sc, 1, L, heads, k);
      s = csa_compress(&sc, 1, L, (const char *)x + r0 * c->d * tb, (const char *)gate + r0 * c->d * tb,
                       (const char *)idx_x + r0 * c->d_idx * tb, (const char *)idx_gate + r0 * c->d_idx * tb,
                       pos_bias, idx_pos_bias, in_dtype, stream);
      if (s) return s;
      s = csa_index_topk(&sc, 1, L, (const char *)q_idx + r0 * heads_idx * c->d_idx * qib, q_idx_dtype,
                         w + r0 * heads_idx, heads_idx, k, idx, cnt, ws, inner_l, stream);
      if (s) return s;
      // every chunk takes the prefill plan (a one-token chunk too): each row is computed alike
      s = attend_common(&sc, 1, L, (const char *)q + r0 * heads * c->d * qb, q_dtype, heads, sink, idx, k,
                        (char *)out + r0 * heads * c->d * ob, out_dtype, out_lse ? out_lse + r0 * heads : nullptr,
                        ws, inner_l, (cudaStream_t)stream, false, true);
      if (s) return s;
    }
  }
  return ok();
}

csa_status csa_static_status(int *status, csa_stream_t stream) {
  if (!status) return fail(CSA_ERR_INVALID_ARG, "NULL pointer");
  csa_status s = CSA_OK;
  void *ws = static_scratch(s);
  if (!ws) return s;
  return csa_device_status(ws, status, stream);
}

csa_status csa_debug_set(int knob, long long value) {
  switch (knob) {
    case CSA_DEBUG_WAIT_LIMIT:
      if (value < 0) return fail(CSA_ERR_INVALID_ARG, "wait limit must be >= 0");
      g_wait_limit.store(value);
      return ok();
    case CSA_DEBUG_STARVE_INDEXER:
      g_starve.store(value != 0);
      return ok();
    default:
      return fail(CSA_ERR_INVALID_ARG, "unknown debug knob %d", knob);
  }
}

csa_status csa_device_status(void *ws, int *status, csa_stream_t stream) {
  if (!ws || !status) return fail(CSA_ERR_INVALID_ARG, "NULL pointer");
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(int), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e, "device status read");
  *status = v;
  return ok();
}

}  // extern "C"
