/*
 * csa.h — C ABI of the B300 (sm_103a) library for DeepSeek-V4 hybrid compressed
 * attention: CSA (compressed sparse attention) and HCA (heavily compressed
 * attention).
 *
 * Sources (web write-ups of the DeepSeek-V4 report), cited by title/section:
 *   [V] "DeepSeek V4 infrastructure" (volanea.com), section "Compression only
 *       works if the attention path is engineered end to end": the CSA parts —
 *       compressed KV entries, lightning-indexer selection, shared key-value
 *       multi-query attention, partial rotary embeddings, sliding-window branch,
 *       attention sink; state caches for the sliding window.
 *   [B] "DeepSeek Releases V4 with Million-Token Context Optimized for AI
 *       Agents" (botbeat.news), section "Summary": 4x compression by
 *       softmax-gated pooling with a learned positional bias plus a lightning
 *       indexer; HCA compresses 128x and attends densely.
 *   [S] "DeepSeek V4: How They Crushed the Million-Token Memory Problem"
 *       (sameershanbhag.com), section "Two kinds of memory instead of one":
 *       ReLU-scored multi-head indexer picking the top-k compressed blocks,
 *       sliding window of uncompressed recent tokens, HCA's dense attention
 *       over 128-token entries, fp8 KV / bf16 rotary dims storage.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All buffers are DEVICE pointers owned by the caller; the library allocates
 *   no memory.  Scratch space is the caller's workspace (csa_workspace_size).
 * - Every call is asynchronous on `stream`.  The return value reports host-side
 *   argument checks and launch errors only; nothing is synchronised.
 * - On error the call launches nothing and csa_last_error() describes it.
 * - Rows of every cache array start on a 16-byte boundary (checked).
 * - A "sequence" b owns n_tokens[b] tokens.  csa_compress appends tokens and
 *   advances n_tokens.  After it, the n_q queries of sequence b sit at
 *   positions n_tokens[b]-n_q .. n_tokens[b]-1 (decode: n_q = 1, t = n_tokens-1).
 * - Entry j of a sequence pools tokens [j*m, (j+1)*m); a query at position t
 *   sees entry j iff (j+1)*m-1 <= t, and window tokens max(0,t-n_win+1) .. t.
 * - Thread safety: calls on distinct workspaces and caches may run concurrently.
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CSA_API __attribute__((visibility("default")))
#else
#define CSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st *csa_stream_t;

typedef int csa_status;
enum {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or dtype */
  CSA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. dims above a limit) */
  CSA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than csa_workspace_size */
  CSA_ERR_CUDA = 4,          /* a CUDA launch failed */
  CSA_ERR_TIMEOUT = 5        /* a device-side bounded wait gave up (csa_device_status) */
};

/*
 * Element types.  CSA_BF16_Q_E4M3 is accepted only as the q_dtype of the indexer
 * calls: the query-side FP8 variant of the lightning indexer ([S] "Two kinds of
 * memory instead of one": the indexer runs in low precision).  The query is
 * passed as bf16; the indexer quantises each (query, head) vector to e4m3 with a
 * power-of-two scale S (max|q_h| * S in [2^7, 2^8), round to nearest even) and
 * scores with q_h' = e4m3(q_h * S) / S.  The default (CSA_BF16) scores with the
 * bf16 query itself.
 */
enum { CSA_F32 = 0, CSA_BF16 = 1, CSA_E4M3 = 2, CSA_BF16_Q_E4M3 = 3, CSA_E2M1 = 4 };

/*
 * One layer's compressed cache.  Geometry fields are host values; pointers are
 * device pointers.  "rows" are physical entry rows:
 *   contiguous (page_size == 0): row(b, j) = b*max_entries + j
 *   paged      (page_size  > 0): row(b, j) = page_table[b*max_pages + j/page_size]*page_size
 *                                            + j%page_size
 * Entry storage ([S]: fp8 for KV, bf16 only for the rotary dims):
 *   kv_dtype == CSA_E4M3: kv_nope u8 e4m3 [rows][d-d_rope], kv_scale f32 [rows],
 *                         kv_rope bf16 [rows][d_rope]; value = code*scale | rope.
 *   kv_dtype == CSA_F32:  kv_nope f32 [rows][d-d_rope], kv_rope f32 [rows][d_rope],
 *                         kv_scale unused (may be NULL).
 * Indexer keys (CSA only, d_idx > 0): idx_key e4m3 [rows][d_idx] + idx_scale f32
 *   [rows] (E4M3) or f32 [rows][d_idx] (F32).  One key per entry, no rotation.
 *   idx_dtype == CSA_E2M1 (FP4 indexer keys, [S]: "FP4 for the indexer"; needs
 *   kv_dtype E4M3 and d_idx in {32, 64, 128}): idx_key u8 [rows][d_idx/2], two OCP
 *   e2m1 codes per byte (element 2i in the low nibble, 2i+1 in the high), idx_scale
 *   f32 [rows]; key = code * scale, scale = max|key|/6 in fp32 (1 if that is 0 or
 *   subnormal), codes rounded to nearest even and saturated at +-6.
 * Stored entries are already rotated (partial RoPE at the block's first token).
 * win: the sliding-window ring [B][win_cap][d] in win_dtype (CSA_F32 or CSA_BF16)
 *   holding RAW (unrotated) recent tokens: token p lives in slot p % win_cap.
 * pool_state: f32 [B][3][d + d_idx]: running (max, sum, weighted sum) of the
 *   softmax-gated pooling of the block in progress; all zeros = empty block.
 * n_tokens: int64 [B] tokens in each sequence (advanced by csa_compress).
 */
typedef struct csa_cache {
  int32_t m;            /* tokens per entry: 4 (CSA), 128 (HCA); 1..1024 */
  int32_t d;            /* KV vector dim incl. rotary dims; multiple of 16, <= 1024-d_idx */
  int32_t d_rope;       /* trailing rotary dims; even, <= 64, <= d */
  int32_t d_idx;        /* indexer key dim (0 = no indexer stream); multiple of 16, <= 128 */
  int32_t kv_dtype;     /* CSA_E4M3 or CSA_F32 */
  int32_t win_dtype;    /* CSA_BF16 or CSA_F32 */
  int32_t n_win;        /* window length W (>= 1) */
  int32_t win_cap;      /* ring slots per sequence (>= W + n_q - 1 for a call with n_q queries) */
  int32_t page_size;    /* entries per page, 0 = contiguous */
  int32_t max_pages;    /* page-table row length (paged) */
  int64_t max_entries;  /* entry capacity per sequence (contiguous) */
  double rope_theta;    /* rotary base, e.g. 10000 */
  void *kv_nope;
  float *kv_scale;
  void *kv_rope;
  void *idx_key;
  float *idx_scale;
  const int32_t *page_table;
  void *win;
  float *pool_state;
  int64_t *n_tokens;
  int32_t idx_dtype;    /* indexer-key storage: 0 = as kv_dtype, CSA_E2M1 = FP4 (see above) */
} csa_cache;

/* Library version (major*10000 + minor*100 + patch). */
CSA_API int csa_version(void);

/* Message of the last failed call on this host thread ("" if none). */
CSA_API const char *csa_last_error(void);

/*
 * Workspace bytes that csa_index_topk, csa_topk, csa_sparse_attend and
 * hca_attend need for `batch` sequences with `n_q` queries each, `heads` query
 * heads and top-k size `k` (k = 0 for HCA).  Alignment: 256 bytes.  The first
 * 256 bytes hold a device status word (see csa_device_status).  For calls of at
 * most 256 query rows with a top-k, the last bytes hold the fused call's top-k
 * area (per-row score-prefix counts, counters and candidate lists); its contents
 * need no initialisation (counts that do not match the scores only cost time)
 * and calls on one workspace must be stream-ordered.
 * Returns 0 when the cache geometry is invalid.
 */
CSA_API size_t csa_workspace_size(const csa_cache *cache, int batch, int n_q, int heads, int k);

/*
 * a1 — compression + append ([B] softmax-gated pooling with a learned positional
 * bias; [S] every 4 (CSA) / 128 (HCA) tokens become one entry; [V] compressed
 * KV entries, partial RoPE; [S] fp8 KV + bf16 rotary dims).
 * Appends n_new tokens to each of `batch` sequences at positions n_tokens[b] ..
 * n_tokens[b]+n_new-1.  For every token: the raw vector is copied into the
 * window ring; the pooling of its block is advanced: per channel c and slot i
 * of the block, logit = gate[c] + pos_bias[i], weights = softmax over the m
 * slots, entry = weighted sum of the token vectors.  When a block completes its
 * entry is rotated (last d_rope dims, position = block's first token), quantised
 * (E4M3: scale = max|nope|/448 in fp32, 1 if that is 0 or subnormal; codes RNE
 * satfinite; rope dims to bf16 RNE) and written at row(b, j).  The indexer-key
 * stream (idx_x, idx_gate, idx_pos_bias; CSA only) is pooled the same way into
 * idx_key (e4m3 with its own scale; not rotated).  n_tokens[b] += n_new.
 *   x, gate        [batch][n_new][d]      in_dtype (must equal cache->win_dtype)
 *   idx_x, idx_gate[batch][n_new][d_idx]  in_dtype (NULL when d_idx == 0)
 *   pos_bias, idx_pos_bias  f32 [m]
 * Requires n_new >= 1; rows of the completed entries must be within capacity.
 */
CSA_API csa_status csa_compress(const csa_cache *cache, int batch, int n_new, const void *x, const void *gate,
                        const void *idx_x, const void *idx_gate, const float *pos_bias,
                        const float *idx_pos_bias, int in_dtype, csa_stream_t stream);

/*
 * a2 — lightning-indexer scores ([S] ReLU-scored multi-head dot products; [V]
 * sparse selection through the indexer).  For query i of sequence b at
 * position t and each visible entry j < (t+1)/m:
 *     scores[(b*n_q + i)*scores_stride + j] = sum_h w[h] * ReLU(q_idx[h] . key_j)
 * with key_j = idx_scale[row]*e4m3(idx_key[row]) (or the f32 key).
 *   q_idx [batch][n_q][heads_idx][d_idx] in q_dtype (CSA_BF16, CSA_F32, or CSA_BF16_Q_E4M3:
 *         bf16 values scored through their e4m3 quantisation, see the element types)
 *   w     f32 [batch][n_q][heads_idx]
 * Entries at or past the visible count are not written.
 */
CSA_API csa_status csa_index_scores(const csa_cache *cache, int batch, int n_q, const void *q_idx, int q_dtype,
                            const float *w, int heads_idx, float *scores, int64_t scores_stride,
                            void *ws, size_t ws_bytes, csa_stream_t stream);

/*
 * a3 — top-k selection ([S] the indexer keeps the top-k compressed blocks).
 * For each query row: the k visible entries with the largest scores, ties to
 * the lower index, written in ascending index order to out_idx[row*k ..];
 * fewer than k visible entries: all of them, then -1 padding.
 * out_count[row] = number of valid indices.  NaN scores are not allowed.
 */
CSA_API csa_status csa_topk(const csa_cache *cache, int batch, int n_q, const float *scores, int64_t scores_stride,
                    int k, int32_t *out_idx, int32_t *out_count, void *ws, size_t ws_bytes,
                    csa_stream_t stream);

/* a2 + a3 in one call; the scores live in the workspace. */
CSA_API csa_status csa_index_topk(const csa_cache *cache, int batch, int n_q, const void *q_idx, int q_dtype,
                          const float *w, int heads_idx, int k, int32_t *out_idx, int32_t *out_count,
                          void *ws, size_t ws_bytes, csa_stream_t stream);

/*
 * a4 — CSA sparse attention ([V] shared key-value multi-query attention,
 * sliding-window branch, attention sink, partial RoPE; [S] window of recent
 * uncompressed tokens).  For query i of sequence b at position t and head h:
 *   q~ = q rotated at t (last d_rope dims); key set = entries idx[row][0..k)
 *   (negative = absent) plus window tokens max(0,t-n_win+1)..t read raw from the
 *   ring and rotated at their positions.  Every key vector is also its value.
 *   l = q~ . kappa / sqrt(d);  out = sum p*kappa with
 *   p = exp(l) / (sum exp(l) + exp(sink[h]));  out_lse = log(sum exp(l) + exp(sink[h])).
 *   q    [batch][n_q][heads][d]  q_dtype (CSA_BF16 or CSA_F32)
 *   sink f32 [heads];  idx int32 [batch][n_q][k]
 *   out  [batch][n_q][heads][d]  out_dtype (CSA_BF16 or CSA_F32);  out_lse f32 [batch][n_q][heads] or NULL
 * heads <= 128, d <= 1024.
 */
CSA_API csa_status csa_sparse_attend(const csa_cache *cache, int batch, int n_q, const void *q, int q_dtype,
                             int heads, const float *sink, const int32_t *idx, int k, void *out,
                             int out_dtype, float *out_lse, void *ws, size_t ws_bytes, csa_stream_t stream);

/*
 * a5 — HCA dense attention ([B] HCA compresses 128x and attends densely; [S]
 * full attention over every compressed entry, same window branch).  As
 * csa_sparse_attend with the key set = all visible entries j < (t+1)/m plus the
 * window and the sink.
 */
CSA_API csa_status hca_attend(const csa_cache *cache, int batch, int n_q, const void *q, int q_dtype, int heads,
                      const float *sink, void *out, int out_dtype, float *out_lse, void *ws,
                      size_t ws_bytes, csa_stream_t stream);

/*
 * Sliding-window-only layer ([S] "Two kinds of memory instead of one": the
 * multi-token-prediction block attends through the sliding window alone): the same
 * shared-KV attention as hca_attend with no compressed entries -- the key set of a
 * query at t is the window tokens max(0, t-n_win+1) .. t (rotated at their
 * positions) plus the sink.  Such a layer's cache needs only its geometry (d,
 * d_rope, n_win, win_cap, win_dtype, rope_theta), win and n_tokens; m, the entry
 * storage and the indexer stream are ignored and may be NULL.
 *   swa_append:  raw tokens x [batch][n_new][d] (in_dtype = win_dtype, 16-byte
 *                aligned) go into the ring; n_tokens[b] += n_new.  No pooling.
 *   swa_attend:  arguments and outputs as hca_attend; the workspace may be NULL
 *                when swa_workspace_size returns 256 or less.
 */
CSA_API size_t swa_workspace_size(const csa_cache *cache, int batch, int n_q, int heads);
CSA_API csa_status swa_append(const csa_cache *cache, int batch, int n_new, const void *x, int in_dtype,
                              csa_stream_t stream);
CSA_API csa_status swa_attend(const csa_cache *cache, int batch, int n_q, const void *q, int q_dtype, int heads,
                              const float *sink, void *out, int out_dtype, float *out_lse, void *ws,
                              size_t ws_bytes, csa_stream_t stream);

/*
 * Prefill of a long prompt in chunks ([E] "Practical Applications": processing
 * million-token inputs): for every sequence b and every chunk of `chunk` new tokens,
 * in order, csa_compress appends the chunk, csa_index_topk selects k entries for
 * each of its queries and csa_sparse_attend attends -- each query sees exactly what
 * a one-shot prefill of all n_new tokens would let it see, and every query row is
 * computed the same way, so the result does not depend on the chunk length.
 * Inputs are [batch][n_new][...] as in the calls above: x, gate [..][d] and idx_x,
 * idx_gate [..][d_idx] in in_dtype; q_idx [..][heads_idx][d_idx] in q_idx_dtype;
 * w f32 [..][heads_idx]; q [..][heads][d] in q_dtype; out [..][heads][d] in
 * out_dtype; out_lse f32 [..][heads] or NULL.  win_cap >= n_win + chunk - 1.
 * The workspace (csa_prefill_workspace_size bytes for this chunk length, 256-byte
 * aligned) holds the calls' scratch -- its status word first -- and the chunk's
 * selected indices.  The calls are launched on `stream` in order; none synchronises.
 */
CSA_API size_t csa_prefill_workspace_size(const csa_cache *cache, int chunk, int heads, int k);
CSA_API csa_status csa_prefill_chunked(const csa_cache *cache, int batch, int n_new, int chunk, const void *x,
                                       const void *gate, const void *idx_x, const void *idx_gate,
                                       const float *pos_bias, const float *idx_pos_bias, int in_dtype,
                                       const void *q_idx, int q_idx_dtype, const float *w, int heads_idx,
                                       const void *q, int q_dtype, int heads, const float *sink, int k, void *out,
                                       int out_dtype, float *out_lse, void *ws, size_t ws_bytes,
                                       csa_stream_t stream);

/*
 * csa_index_topk without a workspace argument, for callers that cannot allocate
 * device memory.  (The paper has no counterpart: this is a deployment variant.)
 * Some hosts hand a library only its input and output buffers: an engine that
 * reserved all device memory for its own pool up front, a plugin interface that
 * exposes no allocator, or a latency-critical loop where cudaMalloc/cudaFree
 * (which can synchronise the device) are not allowed.  This entry point keeps
 * its scratch -- the indexer scores of every query row plus the status word --
 * in one statically sized device array inside the library, so the call itself
 * allocates nothing.
 *   - Capacity: CSA_STATIC_SCRATCH_BYTES.  The call needs 256 bytes plus
 *     batch * n_q * entry capacity * 4 bytes (rounded up to 256); a larger
 *     request returns CSA_ERR_WORKSPACE and launches nothing.
 *   - The array exists once per device for the life of the process, on every
 *     device that loads the library.  The first call on a device looks up the
 *     array's device address (cudaGetSymbolAddress, with that device current);
 *     make that first call before any stream capture.  The address is kept for
 *     the life of the process: after cudaDeviceReset on a device the module is
 *     loaded afresh and the array may move, so this entry point must not be
 *     used on that device again in the same process.
 *   - Device-side failures (a bounded wait of the indexer that gave up) are
 *     reported by csa_static_status; the rows of such a call get out_count = -1.
 *   - All calls share the one array and its contents outlive a call: calls that
 *     may overlap on the GPU (different streams, or devices sharing a context)
 *     race on it.  Serialise them.  The status word is cleared on each call.
 *   - Results are those of csa_index_topk on the same inputs.
 */
#define CSA_STATIC_SCRATCH_BYTES ((size_t)8 << 20)
CSA_API csa_status csa_index_topk_static(const csa_cache *cache, int batch, int n_q, const void *q_idx,
                                         int q_dtype, const float *w, int heads_idx, int k, int32_t *out_idx,
                                         int32_t *out_count, csa_stream_t stream);

/*
 * Reads (synchronously, on `stream`) and clears the device status word at the
 * start of a workspace: 0 = fine, otherwise a CSA_ERR_* code set by a kernel
 * whose bounded wait gave up.  Returns CSA_OK or CSA_ERR_CUDA.
 * The word is sticky: while it is nonzero, every top-k that runs on the workspace
 * (csa_index_topk, csa_topk given the workspace) writes out_count = -1 and -1
 * indices for each row instead of selecting from scores that may be incomplete.
 */
CSA_API csa_status csa_device_status(void *ws, int *status, csa_stream_t stream);

/*
 * The same for the status word of csa_index_topk_static's scratch on the current
 * device (that call clears the word when it starts, so this reports its last run).
 */
CSA_API csa_status csa_static_status(int *status, csa_stream_t stream);

/*
 * Failure injection for tests of the bounded waits (process-wide; not for production
 * use).  The tensor-core indexer's mbarrier waits give up after a number of polls,
 * record CSA_ERR_TIMEOUT in the status word, drain the copies and MMAs already issued,
 * free their tensor memory and return; the context stays usable.
 *   CSA_DEBUG_WAIT_LIMIT:     polls before a wait gives up (0 restores the default, 2^24)
 *   CSA_DEBUG_STARVE_INDEXER: nonzero makes the indexer's producer issue no key copies,
 *                             so the first wait for a key tile runs out (0 restores)
 * Returns CSA_OK or CSA_ERR_INVALID_ARG.
 */
enum { CSA_DEBUG_WAIT_LIMIT = 1, CSA_DEBUG_STARVE_INDEXER = 2 };
CSA_API csa_status csa_debug_set(int knob, long long value);

#ifdef __cplusplus
}
#endif
#endif /* CSA_H_ */
