// Host-side declarations of the kernel launchers (one translation unit each).
#pragma once
#include "common.cuh"

namespace csa {

// Launches kern<<<grid, block, smem, st>>>(args...) with, if cluster > 1, a
// cluster dimension along x, and with programmatic stream serialization when
// built with -DCSA_PDL (see pdl_wait / pdl_trigger).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
#ifdef CSA_PDL
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
#endif
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t launch_compress(const CacheView &c, const RopeTable &rope, int batch, int n_new, int in_dtype,
                            const void *x, const void *gate, const void *ix, const void *ig,
                            const float *pb, const float *ipb, cudaStream_t st);

cudaError_t launch_swa_append(const CacheView &c, int batch, int n_new, int in_dtype, const void *x, cudaStream_t st);

cudaError_t launch_index_generic(const CacheView &c, int batch, int n_q, const void *q_idx, int q_dtype,
                                 const float *w, int heads_idx, float *scores, long long stride,
                                 long long n_cap, cudaStream_t st);

// Test hooks of the tensor-core indexer's bounded waits (failure injection):
// wait_limit = polls before a wait gives up (0: the default, 2^24); starve = 1 makes
// the producer issue no key copies, so the MMA warp's first wait runs out.
struct IndexDebug {
  long long wait_limit;
  int starve;
};

struct TopkArea;
bool index_tc_supported(const CacheView &c, int heads_idx);
size_t index_tc_smem_bytes();
cudaError_t launch_index_tc(const CacheView &c, int batch, int n_q, const void *q_idx, int q_dtype, const float *w,
                            int heads_idx, float *scores, long long stride, int num_sms, int *status,
                            const TopkArea *area, const IndexDebug &dbg, cudaStream_t st);

// Histogram of the top kPrefixBits bits of the order-preserving score keys, one per
// query row: the tensor-core indexer fills it (when given one) while it scores, and
// the top-k reads it to find the bin of the k-th largest score, then zeroes it.
constexpr int kPrefixBits = 13;
constexpr int kPrefixBins = 1 << kPrefixBits;
constexpr int kPrefixRowsMax = 256;   // rows served with prefix histograms (decode-sized calls)
constexpr int kCandMax = 4096;        // threshold-bin keys resolved without a pass over every key

// Row-split top-k of a fused index + top-k call: CTA p of a row takes the row's scores
// [p * kSplitChunk, (p + 1) * kSplitChunk).  Its working area follows the prefix
// histograms in the workspace:
//   ctr   [rows][4]      word 0: CTAs of the row done (the ticket)      } zeroed by the
//   dhist [rows][2048]   next 11 bits of the keys in the threshold bin  } indexer
//   slots [rows][parts]  per CTA: (entries listed or -1, keys above the threshold
//                        bin, keys in it, 0);
//   lists [rows][parts][part_cap] (index, key) entries, each CTA's in index order.
constexpr int kSplitChunk = 8192;
constexpr int kSplitPartsMax = 256;   // entry capacities up to 2M entries
constexpr int kDigitBins = 2048;
struct TopkArea {
  unsigned *hist = nullptr;   // [rows][kPrefixBins]
  unsigned *ctr = nullptr;    // [rows][4], followed by dhist: rows * (4 + kDigitBins) words zeroed together
  unsigned *dhist = nullptr;  // [rows][kDigitBins]
  int4 *slots = nullptr;      // [rows][parts]
  uint2 *lists = nullptr;     // [rows][parts][part_cap]
  int parts = 0, part_cap = 0, rows = 0;
};
// bytes of the area for `rows` rows (0 when the call has too many rows for it), and
// its layout at `base` (256-byte aligned)
size_t topk_area_bytes(int rows, long long n_cap, int k);
TopkArea topk_area(void *base, int rows, long long n_cap, int k);

cudaError_t launch_topk(const CacheView &c, int batch, int n_q, const float *scores, long long stride, int k,
                        int32_t *out_idx, int32_t *out_count, const TopkArea *area, int num_sms, const int *status,
                        cudaStream_t st);

constexpr int kHG = 16;
constexpr int kKC = 32;
struct AttendArgs {
  CacheView c;
  RopeTable rope;
  int n_q, heads, q_dtype, out_dtype;
  const uint8_t *q;
  const float *sink;
  const int32_t *idx;   // nullptr: dense (HCA)
  int k;
  int n_splits, chunks_per_split;
  int keys_per_split;   // chunks_per_split x the running kernel's keys per chunk
  float *part_o, *part_ml;
  uint8_t *out;
  float *out_lse;
  float scale;          // 1/sqrt(d)
};
void attend_plan(int n_q, long long list_cap, int n_win, bool tc, bool wide, int &n_splits, int &cps);
bool attend_tc_supported(const CacheView &c, int heads, int q_dtype);
size_t attend_tc_smem_bytes(int d);
cudaError_t launch_attend_tc(const AttendArgs &a, int rows, cudaStream_t st);
size_t attend_smem_bytes(int d);
cudaError_t launch_attend(const AttendArgs &a, int rows, cudaStream_t st);
cudaError_t launch_attend_combine(const AttendArgs &a, int rows, cudaStream_t st);

}  // namespace csa
