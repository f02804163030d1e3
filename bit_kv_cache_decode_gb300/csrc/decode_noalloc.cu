// Decode attention that allocates no device memory (sm_103a).
//
// Some callers cannot call cudaMalloc: serving engines whose allocator already
// owns all device memory and forbids side allocations, and hosts that may not
// allocate on a latency-critical path (cudaMalloc can synchronise the device).
// oscar_decode_attention needs a caller-allocated workspace for its scratch
// (rotated queries, query fragments and sums, split partials, status word);
// this entry point runs the same kernels with that scratch taken from a fixed
// static device array instead.
#include <mutex>

#include "kernels.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;   // 4 MiB per device
constexpr int kMaxDevices = 64;

// The scratch itself. Every GPU that loads the library holds it until the
// process exits. In host code this name is only a stand-in for the symbol;
// kernels get the device address resolved below.
static __device__ __align__(256) uint8_t g_decode_scratch[kScratchBytes];

std::mutex g_mu;
uint8_t* g_addr[kMaxDevices];
int g_sms[kMaxDevices];

// Once per device, with that device current: resolve the array's device address.
int scratch_for_current_device(uint8_t** addr, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OSCAR_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return OSCAR_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return OSCAR_ERR_CUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return OSCAR_ERR_CUDA;
    g_sms[dev] = n;
    g_addr[dev] = static_cast<uint8_t*>(p);
  }
  *addr = g_addr[dev];
  *sms = g_sms[dev];
  return OSCAR_OK;
}

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" int oscar_decode_attention_noalloc(const oscar_layout* layout, void* pool, int layer, int B,
                                              const void* q, const int32_t* seq_lens, const int32_t* hist_pt,
                                              int max_hist_pages, const int32_t* bf16_pt, float sm_scale, void* out,
                                              int out_dtype, float* lse, int* status, void* stream) {
  using namespace oscar;
  if (!layout || !pool || B < 0 || max_hist_pages < 0) return OSCAR_ERR_INVALID_ARG;
  if (out_dtype != OSCAR_OUT_BF16 && out_dtype != OSCAR_OUT_FP32) return OSCAR_ERR_INVALID_ARG;
  if (B == 0) return OSCAR_OK;
  if (!q || !seq_lens || !bf16_pt || !out || (max_hist_pages > 0 && !hist_pt)) return OSCAR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(q) % 16) return OSCAR_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || sm_scale == INFINITY) return OSCAR_ERR_INVALID_ARG;
  LayerView lv;
  int rc = pool_layer_view(layout, pool, layer, nullptr, &lv);
  if (rc != OSCAR_OK) return rc;
  // scratch carving: status word | rotated queries | query fragments | query group sums | partials
  const size_t hq = layout->num_q_heads, hkv = layout->num_kv_heads;
  const size_t fixed = 256 + up256((size_t)B * hq * kD * sizeof(float)) +
                       up256((size_t)B * hkv * kFragWords * sizeof(uint32_t)) +
                       up256((size_t)B * hq * kQConst * sizeof(float));
  const size_t per_slot = (size_t)B * hq * kPartFloats * sizeof(float);
  const int nbf = (layout->sink + layout->recent) / kP;
  // layout: fixed part | partials
  if (fixed + (size_t)partial_slots(1, nbf) * per_slot > kScratchBytes) return OSCAR_ERR_TOO_LARGE;
  rc = configure_kernels();
  if (rc != OSCAR_OK) return rc;
  uint8_t* scratch = nullptr;
  int sms = 0;
  rc = scratch_for_current_device(&scratch, &sms);
  if (rc != OSCAR_OK) return rc;
  const int max_slots = (int)((kScratchBytes - fixed) / per_slot);
  // largest split count whose slots (splits, then BF16 pages) fit
  int max_splits = 1;
  while (max_splits < kMaxMmaSplits && partial_slots(max_splits + 1, nbf) <= max_slots) ++max_splits;
  DecodeWorkspace ws;
  uint8_t* p = scratch;
  int* dstatus = reinterpret_cast<int*>(p);
  p += 256;
  ws.qrot = reinterpret_cast<float*>(p);
  p += up256((size_t)B * hq * kD * sizeof(float));
  ws.qfrag = reinterpret_cast<uint32_t*>(p);
  p += up256((size_t)B * hkv * kFragWords * sizeof(uint32_t));
  ws.qconst = reinterpret_cast<float*>(p);
  p += up256((size_t)B * hq * kQConst * sizeof(float));
  ws.partials = reinterpret_cast<float*>(p);
  ws.cta_trace = nullptr;
  ws.trace_cap = 0;
  lv.status = dstatus;
  DecodeArgs a;
  a.B = B;
  a.q = q;
  a.seq_lens = seq_lens;
  a.hist_pt = hist_pt;
  a.max_hist_pages = max_hist_pages;
  a.bf16_pt = bf16_pt;
  a.sm_scale = sm_scale;
  a.out = out;
  a.out_dtype = out_dtype;
  a.lse = lse;
  a.algo = resolve_decode_algo(kDefaultDecodeAlgo, layout->meta_format, (int)(hq / hkv));
  a.len_add = 0;
  a.skip_qprep = 0;
  a.ev0 = a.ev1 = nullptr;
  a.nbf = nbf;
  decode_split_policy(B, (int)hkv, (int)(hq / hkv), nbf, max_hist_pages, max_splits, sms, a.algo, &a.nsplit,
                      &a.pages_per_split, &a.mma_occupancy);
  ws.max_splits = a.nsplit;
  ws.nslots = partial_slots(a.nsplit, nbf);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: the status word must start at zero
  if (cudaMemsetAsync(dstatus, 0, sizeof(int), st) != cudaSuccess) return OSCAR_ERR_CUDA;
  rc = launch_decode(lv, ws, a, st);
  if (rc != OSCAR_OK) return rc;
  if (status && cudaMemcpyAsync(status, dstatus, sizeof(int), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return OSCAR_ERR_CUDA;
  return OSCAR_OK;
}
