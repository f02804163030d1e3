// Host-side launch interface of the OSCAR kernels (sm_103a).
#pragma once

#include "common.cuh"

namespace oscar {

constexpr int kDefaultDecodeAlgo = OSCAR_DECODE_MMA;
constexpr int kMaxMmaSplits = 2048;        // history splits of the fused decode
// History pages one split of the tensor-core decode covers, at most (16 per
// warp). The tensor cores' fp32 accumulation truncates instead of rounding, so
// its error grows with the number of MMAs summed into one accumulator; longer
// contexts take more splits, whose partials the merge adds with rounding.
constexpr int kMaxPagesPerMmaSplit = 64;
// a BF16 page folded into a history CTA of the fused decode costs about this many history pages of
// that CTA's time (its bulk copies, waited on after the history loop, and its tensor-core products:
// about 4 us on the 102,400-token Qwen3-8B layer, where a CTA's warps take some 2 us per page)
constexpr int kBf16FoldPages = 8;
// partial slots per (request, q head): history splits, then one per BF16 page
inline int partial_slots(int max_splits, int nbf) { return max_splits + nbf; }
constexpr int kPrefillTok = 1024;                                  // tokens per prefill CTA

// Decode workspace carved from the caller's workspace buffer.
struct DecodeWorkspace {
  float* qrot;        // [max_batch][hq][kD] rotated queries (float32, rotated channel order)
  uint32_t* qfrag;    // [max_batch][hkv][kFragWords] fp16 MMA B fragments of the rotated queries
  float* qconst;      // [max_batch][hq][kQConst] per-query-head constants, see kQ* below
  float* partials;    // [max_batch][hq][nslots][kPartFloats]: history splits, then BF16 chunks
  unsigned long long* cta_trace;  // optional per-CTA timeline of the fused decode (see oscar_trace_ctas)
  int trace_cap;      // records available in cta_trace
  int max_splits;     // history splits available
  int nslots;         // partial slots per (request, q head) = max_splits + BF16 chunks
};

// Per-query-head constants written by the query prologue.
constexpr int kQConst = 12;
constexpr int kQSum0 = 0, kQSum1 = 1;    // sum of the rotated query over group 0 / 1
constexpr int kQF = 2;                   // sm_scale * log2(e) * 2^-sigma (fragment scale undo)
constexpr int kQZ0 = 3, kQZ1 = 4;        // sm_scale * log2(e) * group sums (zero-point terms)
constexpr int kQOff0H = 5, kQOff0L = 6;  // 1024 * sum of group 0's fragment values, high and low parts
constexpr int kQOff1H = 7, kQOff1L = 8;  // same for group 1
constexpr int kQSigma = 9;               // sigma, the power-of-two scale of the fragments

// B fragments of one kv head's query group for the tensor-core decode:
// 8 k-blocks x 2 n-tiles x 32 lanes x 2 registers.
constexpr int kFragWords = 8 * 2 * 32 * 2;

int launch_pack_rotated(const LayerView& lv, int kind, const float* xrot, const int* page_ids, const int* rows,
                        int N, cudaStream_t st);
int launch_rotate(const LayerView& lv, int kind, const void* x, float* y, int N, cudaStream_t st);
int launch_prefill(const LayerView& lv, int B, const void* k, const void* v, const int* cu_seqlens, int total,
                   const int* hist_pt, int max_hist_pages, const int* bf16_pt, cudaStream_t st);
// fused projection + write path: K = x W_k^T, V = x W_v^T (bf16), placed and quantised like launch_prefill
int launch_project_prefill(const LayerView& lv, int B, const void* x, int d_model, const void* w_k, const void* w_v,
                           const int* cu_seqlens, int total, const int* hist_pt, int max_hist_pages,
                           const int* bf16_pt, cudaStream_t st);
int configure_project_prefill_kernel();
// Append (k, v non-null: new tokens, demotion) and / or the decode's query prologue (q non-null) in one
// launch, a programmatic dependent of the kernel before it (prologue.cu).
int launch_prologue(const LayerView& lv, const DecodeWorkspace& ws, int B, const void* q, const void* k,
                    const void* v, const int* seq_lens_before, const int* hist_pt, int max_hist_pages,
                    const int* bf16_pt, float sm_scale, cudaStream_t st);
int configure_prologue_kernel();
int configure_write_path_kernels();
int configure_prefill_kernel();   // prefill_tc.cu

struct DecodeArgs {
  int B;
  const void* q;
  const int* seq_lens;
  const int* hist_pt;
  int max_hist_pages;
  const int* bf16_pt;
  float sm_scale;
  void* out;
  int out_dtype;
  float* lse;
  int nsplit;            // history splits launched per (request, kv head)
  int nbf;               // BF16 (sink + recent) chunks of 64 tokens per (request, kv head)
  int pages_per_split;   // history pages per split, at most (the tensor-core path spreads a request evenly)
  int shared_pages = 0;  // tensor-core path: history pages [0, shared_pages) are the same for every request
  int nsplit_shared = 0; // splits of the shared pages per kv head (their slots follow the nsplit history slots)
  int mma_occupancy = 3; // tensor-core path, gq <= 4: resident CTAs per SM of the decode kernel variant (3 or 4)
  int algo;              // OSCAR_DECODE_SIMT / OSCAR_DECODE_MMA
  int len_add;           // the kernels attend over seq_lens[b] + len_add tokens
  int skip_qprep;        // the query prologue already ran (with the append, in one launch)
  cudaEvent_t ev0, ev1;  // optional events around the history (fused decode) kernel, may be null
};

int launch_decode(const LayerView& lv, const DecodeWorkspace& ws, const DecodeArgs& a, cudaStream_t st);
// tcgen05 decode (decode_tc.cu): the history splits and, in one more CTA per (request, kv head), the
// BF16 pages; the layouts it serves (fp16 metadata, gq <= 4)
bool decode_tc_supported(const LayerView& lv);
int launch_decode_tc(const LayerView& lv, const DecodeWorkspace& ws, const DecodeArgs& a, float scale_log2,
                     cudaStream_t st);
int configure_tc_kernel();
// the decode kernel that runs for a requested algorithm: OSCAR_DECODE_TC only where the tcgen05 kernel
// serves the layout (fp16 metadata, up to 4 query heads per kv head), else OSCAR_DECODE_MMA
inline int resolve_decode_algo(int algo, int meta_format, int gq) {
  if (algo == OSCAR_DECODE_TC && (meta_format != OSCAR_META_F16 || gq > 4)) return OSCAR_DECODE_MMA;
  return algo;
}
// Merge of the partial slots of every (request, q head): history slots [0, nsplit),
// BF16 slots [nsplit, nsplit + nbfs). Launched as a programmatic dependent of the
// kernel that wrote the partials.
int launch_merge(const LayerView& lv, const DecodeWorkspace& ws, int B, int nsplit, int nbfs, void* out,
                 int out_dtype, float* lse, cudaStream_t st);
constexpr int kMergeChunk = 96;            // partial slots staged in shared memory at a time by the merge
int configure_merge_kernel();
constexpr int kSharedRows = 128;   // query rows (request x head) per CTA of the shared-prefix decode
int launch_decode_shared(const LayerView& lv, const DecodeWorkspace& ws, const DecodeArgs& a, cudaStream_t st);
int configure_shared_kernel();

// The kernels of the decode chain all ask for the largest shared-memory carveout: a grid scheduled
// early beside its predecessor then never waits for an SM to drain and change its L1 / shared split.
inline int set_max_shared_carveout(const void* fn) {
  return cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared) == cudaSuccess
             ? OSCAR_OK
             : OSCAR_ERR_CUDA;
}
int configure_decode_kernels();
int launch_wait_probe(int* status, cudaStream_t st);   // checks.cu

// the streaming BF16 comparison kernel (bf16_decode.cu): partials of `nsplit` splits of pages_per_split pages
int launch_bf16_stream(int B, int hkv, int hq, const void* kv_pages, int num_pages, const void* q,
                       const int* seq_lens, const int* page_table, int max_pages, int pages_per_split, int nsplit,
                       float scale_log2, float* partials, int nslots, int* status, cudaStream_t st);
int configure_bf16_stream();
int launch_bf16_decode(int B, int hq, int hkv, const void* kv_pages, int num_pages, const void* q,
                       const int* seq_lens, const int* page_table, int max_pages, float sm_scale, void* out,
                       int out_dtype, float* lse, float* partials, int max_splits, int nsplit, int pages_per_split,
                       int* status, cudaStream_t st);

}  // namespace oscar

namespace oscar {
// api.cu helpers for entry points that work without a cache handle
int pool_layer_view(const oscar_layout* L, void* pool, int layer, int* status, LayerView* out);
void decode_split_policy(int B, int hkv, int gq, int nbf, int max_pages, int max_splits, int sms, int algo,
                         int* nsplit, int* pps, int* occupancy);
int configure_kernels();
}  // namespace oscar
