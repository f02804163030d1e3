// C ABI of the OSCAR INT2 KV-cache library: layout carving, argument checks,
// launches, status and tracing. The functions and data layouts are described
// in include/oscar.h.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "kernels.cuh"

using namespace oscar;

struct oscar_cache {
  oscar_layout lay;
  uint8_t* pool;
  uint8_t* ws;
  size_t layer_bytes, int2_bytes, bf16_bytes, params_bytes;
  size_t pool_bytes, ws_bytes;
  DecodeWorkspace dws;
  int* status;
  int sms;
  int algo;
  unsigned long long* timeline;   // kernel timeline buffer (oscar_trace_timeline) or null
  int timeline_cap;
  // tracing
  bool prof_on;
  int prof_cap, prof_n;
  std::vector<cudaEvent_t> prof_ev;
};

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool is_pow2_le8(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

int check_layout(const oscar_layout* L) {
  if (!L) return OSCAR_ERR_INVALID_ARG;
  if (L->num_layers < 1 || L->num_kv_heads < 1 || L->num_q_heads < 1 || L->num_int2_pages < 0 ||
      L->num_bf16_pages < 0 || L->max_batch < 1 || L->max_splits < 1 || L->sink < 0 || L->recent < 1)
    return OSCAR_ERR_INVALID_ARG;
  if (L->num_q_heads % L->num_kv_heads != 0) return OSCAR_ERR_INVALID_ARG;
  if (L->page_size < 1 || L->sink % L->page_size != 0 || L->recent % L->page_size != 0) return OSCAR_ERR_INVALID_ARG;
  if (L->group < 1 || L->head_dim % L->group != 0) return OSCAR_ERR_INVALID_ARG;
  if (L->v_mode != OSCAR_V_ABSORBED && L->v_mode != OSCAR_V_EXPLICIT) return OSCAR_ERR_INVALID_ARG;
  if (L->meta_format != OSCAR_META_F16 && L->meta_format != OSCAR_META_U8 && L->meta_format != OSCAR_META_CB)
    return OSCAR_ERR_INVALID_ARG;
  if (L->head_dim != kD || L->group != kG || L->page_size != kP) return OSCAR_ERR_UNSUPPORTED;
  if (!is_pow2_le8(L->num_q_heads / L->num_kv_heads)) return OSCAR_ERR_UNSUPPORTED;
  if (L->max_splits > 4096) return OSCAR_ERR_UNSUPPORTED;
  return OSCAR_OK;
}

void sizes(const oscar_layout* L, size_t* int2b, size_t* bf16b, size_t* prmb, size_t* layerb, size_t* poolb,
           size_t* wsb) {
  *int2b = align_up((size_t)L->num_int2_pages * L->num_kv_heads *
                    (L->meta_format == OSCAR_META_U8 ? kBlockBytesU8 : kBlockBytes));
  *bf16b = align_up((size_t)L->num_bf16_pages * L->num_kv_heads * kBf16BlockBytes);
  *prmb = align_up((size_t)L->num_kv_heads * kParamFloats * sizeof(float));
  *layerb = *int2b + *bf16b + *prmb;
  *poolb = *layerb * L->num_layers;
  const size_t B = L->max_batch, hq = L->num_q_heads, hkv = L->num_kv_heads;
  *wsb = kAlign                                                    // status word
         + align_up(B * hq * kD * sizeof(float))                   // qrot
         + align_up(B * hkv * kFragWords * sizeof(uint32_t))       // qfrag
         + align_up(B * hq * kQConst * sizeof(float))              // qconst
         + align_up(B * hq * partial_slots(L->max_splits, (L->sink + L->recent) / kP) * kPartFloats * sizeof(float));
}

LayerView view(const oscar_cache* c, int layer) {
  LayerView v;
  uint8_t* base = c->pool + (size_t)layer * c->layer_bytes;
  v.int2 = base;
  v.bf16 = base + c->int2_bytes;
  v.params = reinterpret_cast<const float*>(base + c->int2_bytes + c->bf16_bytes);
  v.next_params = layer + 1 < c->lay.num_layers ? reinterpret_cast<const float*>(
                                                      reinterpret_cast<const uint8_t*>(v.params) + c->layer_bytes)
                                                : nullptr;
  v.n_int2 = c->lay.num_int2_pages;
  v.n_bf16 = c->lay.num_bf16_pages;
  v.hkv = c->lay.num_kv_heads;
  v.hq = c->lay.num_q_heads;
  v.sink = c->lay.sink;
  v.recent = c->lay.recent;
  v.v_explicit = c->lay.v_mode == OSCAR_V_EXPLICIT;
  v.meta_u8 = c->lay.meta_format == OSCAR_META_U8;
  v.meta_cb = c->lay.meta_format == OSCAR_META_CB;
  v.blk_bytes = v.meta_u8 ? kBlockBytesU8 : kBlockBytes;
  v.status = c->status;
  v.layer = layer;
  v.timeline = c->timeline;
  v.timeline_cap = c->timeline_cap;
  return v;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// R = U H P_br (MarkTechPost article "Together AI 开源 OSCAR…", section "OSCAR 有何不同做法"), composed in
// double from the float32 U as loaded: (U H)[i][c] = sum_m U[i][m] (-1)^popcount(m & c) / sqrt(128), and
// column j of R is column bitrev7(j) of U H. R[i][j]: i = input channel, j = rotated channel.
std::vector<double> composite_rotation(const float* U) {
  std::vector<double> uh((size_t)kD * kD), R((size_t)kD * kD);
  const double inv = 1.0 / std::sqrt((double)kD);
  for (int i = 0; i < kD; ++i)
    for (int c = 0; c < kD; ++c) {
      double s = 0.0;
      for (int m = 0; m < kD; ++m) s += (double)U[i * kD + m] * ((__builtin_popcount(m & c) & 1) ? -inv : inv);
      uh[(size_t)i * kD + c] = s;
    }
  for (int j = 0; j < kD; ++j) {
    int rj = 0;
    for (int bit = 0; bit < 7; ++bit) rj |= ((j >> bit) & 1) << (6 - bit);
    for (int i = 0; i < kD; ++i) R[(size_t)i * kD + j] = uh[(size_t)i * kD + rj];
  }
  return R;
}

// R as fp16 hi = fp16(R), lo = fp16(R - hi) (about 22 significant bits) in the B-fragment order of
// mma.m16n8k16 (k = input channel, n = rotated channel): for k-block kb, n-tile nt and lane (g = lane / 4,
// t = lane % 4), b0 holds rows 16 kb + 2t, +1 and b1 rows 16 kb + 2t + 8, +9, all of column 8 nt + g.
void rotation_fragments(const std::vector<double>& R, uint32_t* frag) {
  auto half_bits = [](double x) -> uint32_t {
    const __half hv = __double2half(x);
    return (uint32_t)__half_as_ushort(hv);
  };
  auto half_val = [](double x) -> double { return (double)__half2float(__double2half(x)); };
  for (int kb = 0; kb < 8; ++kb)
    for (int nt = 0; nt < 16; ++nt)
      for (int lane = 0; lane < 32; ++lane) {
        const int g = lane >> 2, t = lane & 3, col = 8 * nt + g;
        const int rows[4] = {16 * kb + 2 * t, 16 * kb + 2 * t + 1, 16 * kb + 2 * t + 8, 16 * kb + 2 * t + 9};
        uint32_t hi[4], lo[4];
        for (int e = 0; e < 4; ++e) {
          const double r = R[(size_t)rows[e] * kD + col];
          hi[e] = half_bits(r);
          lo[e] = half_bits(r - half_val(r));
        }
        uint32_t* w = frag + (((size_t)kb * 16 + nt) * 32 + lane) * 4;
        w[0] = hi[0] | (hi[1] << 16);
        w[1] = hi[2] | (hi[3] << 16);
        w[2] = lo[0] | (lo[1] << 16);
        w[3] = lo[2] | (lo[3] << 16);
      }
}

// R as three bf16 parts b1 = bf16(R), b2 = bf16(R - b1), b3 = bf16(R - b1 - b2), each laid out as the
// bulk prefill's tensor-core B operand (n = rotated channel, k = input channel, K-major, 128-byte swizzle):
// element (n, k) of part p at byte p * 32768 + (k / 64) * 16384 + n * 128 + (((k % 64) / 8) ^ (n % 8)) * 16
// + (k % 8) * 2.
void rotation_image(const std::vector<double>& R, uint8_t* img) {
  auto bf16_bits = [](double x) -> uint16_t {
    const __nv_bfloat16 b = __float2bfloat16_rn((float)x);
    return *reinterpret_cast<const uint16_t*>(&b);
  };
  auto bf16_val = [](uint16_t bits) -> double {
    const uint32_t w = (uint32_t)bits << 16;
    float f;
    std::memcpy(&f, &w, 4);
    return (double)f;
  };
  for (int n = 0; n < kD; ++n)
    for (int k = 0; k < kD; ++k) {
      double r = R[(size_t)k * kD + n];
      const size_t off = (size_t)(k >> 6) * 16384 + (size_t)n * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) + (k & 7) * 2;
      for (int p = 0; p < 3; ++p) {
        const uint16_t b = bf16_bits(r);
        std::memcpy(img + (size_t)p * 32768 + off, &b, 2);
        r -= bf16_val(b);
      }
    }
}

// Kernel attributes (dynamic shared memory limits, carveout) belong to one device's context: they are
// set once per device, the first time a call needs the kernels on that device.
constexpr int kMaxConfiguredDevices = 64;
std::mutex g_configure_mu;
bool g_configured[kMaxConfiguredDevices];

int configure_once() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OSCAR_ERR_CUDA;
  if (dev < 0 || dev >= kMaxConfiguredDevices) return OSCAR_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_configure_mu);
  if (g_configured[dev]) return OSCAR_OK;
  int rc = configure_write_path_kernels();
  if (rc == OSCAR_OK) rc = configure_decode_kernels();
  if (rc == OSCAR_OK) g_configured[dev] = true;
  return rc;
}

// CUDA-core split policy over the page-table width: the number of history
// splits per (request, kv head) that minimises waves x (pages per CTA + a fixed
// per-CTA cost), where a wave is sms * ctas_per_sm resident CTAs; there is no
// empty trailing split.
void choose_splits_simt(int B, int hkv, int max_pages, int max_splits, int sms, int* nsplit, int* pps) {
  if (max_pages <= 0) { *nsplit = 1; *pps = 1; return; }
  const long units = (long)B * hkv, slots = std::max(1L, (long)sms * 4);
  const int nmax = std::min(std::min(max_splits, max_pages), kMaxMmaSplits);
  long best_cost = -1;
  int best_p = max_pages;
  for (int n = 1; n <= nmax; ++n) {
    const int p = (max_pages + n - 1) / n;
    const int used = (max_pages + p - 1) / p;
    const long waves = (units * used + slots - 1) / slots;
    const long cost = waves * (p + 2L);
    if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_p = p; }
  }
  *pps = best_p;
  *nsplit = (max_pages + best_p - 1) / best_p;
}

// tcgen05 split policy. Two history CTAs fit an SM (TMEM and registers); one more CTA per (request, kv
// head) takes the BF16 pages and the step prologue holds about half a CTA's registers per (request, kv
// head, K / V) while the decode is scheduled. The history CTAs fill the remaining slots of one wave,
// each taking at least one tile of two pages and at most 256 pages (the output accumulates in TMEM over
// a split; longer contexts take more splits).
void choose_splits_tc(int B, int hkv, int max_pages, int max_splits, int sms, int* nsplit, int* pps) {
  if (max_pages <= 0) { *nsplit = 1; *pps = 1; return; }
  const long units = (long)B * hkv;
  const long budget = 2L * sms - units - std::min((long)sms, units);
  int n = (int)std::max(1L, budget / std::max(1L, units));
  n = std::max(n, (max_pages + 255) / 256);
  n = std::min(n, std::max(1, max_pages / 2));
  n = std::min(std::min(n, max_splits), kMaxMmaSplits);
  *nsplit = std::max(1, n);
  *pps = (max_pages + *nsplit - 1) / *nsplit;
}

// Tensor-core split policy. A request's history pages are spread over n splits of 4 warps, a warp
// taking every fourth page of its split. With n >= nbf the BF16 pages fold into the last nbf splits,
// each kBf16FoldPages history pages lighter for it: the grid has B * hkv * n CTAs, all about equally
// heavy, so the SMs finish together whichever CTAs they hold. With fewer splits each BF16 page takes a
// light CTA of its own (B * hkv * (n + nbf) CTAs). ctas_per_sm are resident per SM. The kernel is
// issue-bound, so an SM's time follows the pages it holds: n minimises waves x (pages per warp, as a
// fraction, + 2 rounds of per-CTA cost: the first page's latency, the warps' combine, one more merge
// slot), with at most kMaxPagesPerMmaSplit pages per split when the split budget allows. The step
// prologue, which runs as the decode is scheduled (2 CTAs per request and kv head), holds one decode
// CTA's registers on each SM it occupies: the first wave has that many fewer slots.
void choose_splits_mma(int B, int hkv, int gq, int nbf, int max_pages, int max_splits, int sms, int* nsplit,
                       int* pps, int* occupancy) {
  *occupancy = gq <= 4 ? 3 : 2;                      // the kernel variants' resident CTAs per SM
  if (max_pages <= 0) { *nsplit = 1; *pps = 1; return; }
  const long units = (long)B * hkv, reserved = std::min((long)sms, 2 * units);
  const int nmax = std::min(std::min(max_splits, max_pages), kMaxMmaSplits);
  auto best = [&](int ctas_per_sm, long* waves_out) {
    const long slots = std::max(1L, (long)sms * ctas_per_sm);
    double best_cost = -1.0;
    int best_n = nmax;
    long best_waves = 1;
    for (int n = 1; n <= nmax; ++n) {
      const bool fold = n >= nbf;
      const int per = fold ? (max_pages + nbf * kBf16FoldPages + n - 1) / n : (max_pages + n - 1) / n;
      if (per > kMaxPagesPerMmaSplit && n < nmax) continue;
      const long ctas = units * (fold ? n : n + nbf);
      const long waves = std::max(1L, (ctas + reserved + slots - 1) / slots);
      const double cost = (double)waves * (per / 4.0 + 2.0);   // issue-bound: an SM's pages, not its slowest warp
      if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_n = n; best_waves = waves; }
    }
    *waves_out = best_waves;
    return best_n;
  };
  long waves = 1;
  int n = best(*occupancy, &waves);
  if (gq <= 4 && waves > 2) {                        // many waves: the 4-CTA variant hides latency better
    *occupancy = 4;
    n = best(4, &waves);
  }
  *nsplit = n;
  *pps = (max_pages + n - 1) / n;
}

// Codebook levels and decision thresholds as the kernels read them: k_i as floats, then
// theta_i = fl32((k_i + k_{i+1}) / 510).
void codebook_consts(const uint8_t* k, float* out) {
  for (int i = 0; i < 4; ++i) out[i] = (float)k[i];
  for (int i = 0; i < 3; ++i) out[4 + i] = (float)(k[i] + k[i + 1]) / 510.0f;
  out[7] = 0.f;
}

}  // namespace

extern "C" {

const char* oscar_error_string(int code) {
  switch (code) {
    case OSCAR_OK: return "ok";
    case OSCAR_ERR_INVALID_ARG: return "invalid argument";
    case OSCAR_ERR_UNSUPPORTED: return "unsupported shape or mode";
    case OSCAR_ERR_CUDA: return "CUDA runtime error";
    case OSCAR_ERR_DEVICE_STATUS: return "device status word has error bits";
    case OSCAR_ERR_TIMEOUT: return "bounded device wait expired";
    case OSCAR_ERR_NOT_ORTHOGONAL: return "rotation is not orthogonal (max|U^T U - I| > 1e-3)";
    case OSCAR_ERR_TOO_LARGE: return "call needs more than the fixed device scratch of the allocation-free decode";
    default: return "unknown status";
  }
}

int oscar_cache_bytes(const oscar_layout* layout, size_t* pool_bytes, size_t* workspace_bytes) {
  int rc = check_layout(layout);
  if (rc != OSCAR_OK) return rc;
  size_t a, b, c, d, pb, wb;
  sizes(layout, &a, &b, &c, &d, &pb, &wb);
  if (pool_bytes) *pool_bytes = pb;
  if (workspace_bytes) *workspace_bytes = wb;
  return OSCAR_OK;
}

int oscar_cache_create(const oscar_layout* layout, void* pool, void* workspace, oscar_cache** out) {
  if (!out) return OSCAR_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = check_layout(layout);
  if (rc != OSCAR_OK) return rc;
  if (!pool || !workspace) return OSCAR_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(pool) | reinterpret_cast<uintptr_t>(workspace)) % kAlign != 0)
    return OSCAR_ERR_INVALID_ARG;
  rc = configure_once();
  if (rc != OSCAR_OK) return rc;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OSCAR_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return OSCAR_ERR_CUDA;
  oscar_cache* c = new (std::nothrow) oscar_cache();
  if (!c) return OSCAR_ERR_INVALID_ARG;
  c->lay = *layout;
  c->pool = static_cast<uint8_t*>(pool);
  c->ws = static_cast<uint8_t*>(workspace);
  sizes(layout, &c->int2_bytes, &c->bf16_bytes, &c->params_bytes, &c->layer_bytes, &c->pool_bytes, &c->ws_bytes);
  const size_t B = layout->max_batch, hq = layout->num_q_heads, hkv = layout->num_kv_heads;
  uint8_t* p = c->ws;
  c->status = reinterpret_cast<int*>(p);
  p += kAlign;
  c->dws.qrot = reinterpret_cast<float*>(p);
  p += align_up(B * hq * kD * sizeof(float));
  c->dws.qfrag = reinterpret_cast<uint32_t*>(p);
  p += align_up(B * hkv * kFragWords * sizeof(uint32_t));
  c->dws.qconst = reinterpret_cast<float*>(p);
  p += align_up(B * hq * kQConst * sizeof(float));
  c->dws.partials = reinterpret_cast<float*>(p);
  c->dws.max_splits = layout->max_splits;
  c->dws.cta_trace = nullptr;
  c->dws.trace_cap = 0;
  c->dws.nslots = partial_slots(layout->max_splits, (layout->sink + layout->recent) / kP);
  p += align_up(B * hq * c->dws.nslots * kPartFloats * sizeof(float));
  c->sms = sms;
  c->algo = kDefaultDecodeAlgo;
  c->timeline = nullptr;
  c->timeline_cap = 0;
  c->prof_on = false;
  c->prof_cap = c->prof_n = 0;
  if (cudaMemset(c->status, 0, sizeof(int)) != cudaSuccess) {
    delete c;
    return OSCAR_ERR_CUDA;
  }
  *out = c;
  return OSCAR_OK;
}

int oscar_cache_destroy(oscar_cache* c) {
  if (!c) return OSCAR_OK;
  for (cudaEvent_t e : c->prof_ev) cudaEventDestroy(e);
  delete c;
  return OSCAR_OK;
}

int oscar_layer_offsets(const oscar_cache* c, int layer, size_t* int2_off, size_t* bf16_off, size_t* params_off) {
  if (!c || layer < 0 || layer >= c->lay.num_layers) return OSCAR_ERR_INVALID_ARG;
  const size_t base = (size_t)layer * c->layer_bytes;
  if (int2_off) *int2_off = base;
  if (bf16_off) *bf16_off = base + c->int2_bytes;
  if (params_off) *params_off = base + c->int2_bytes + c->bf16_bytes;
  return OSCAR_OK;
}

int oscar_set_codebook(oscar_cache* c, int layer, const uint8_t* cb_K, const uint8_t* cb_V, void* stream) {
  if (!c || layer < 0 || layer >= c->lay.num_layers || !cb_K || !cb_V) return OSCAR_ERR_INVALID_ARG;
  if (c->lay.meta_format != OSCAR_META_CB) return OSCAR_ERR_UNSUPPORTED;
  const int hkv = c->lay.num_kv_heads;
  for (int h = 0; h < hkv; ++h)
    for (int i = 0; i < 3; ++i)
      if (cb_K[4 * h + i] > cb_K[4 * h + i + 1] || cb_V[4 * h + i] > cb_V[4 * h + i + 1]) return OSCAR_ERR_INVALID_ARG;
  LayerView v = view(c, layer);
  std::vector<float> host((size_t)hkv * 16, 0.f);
  for (int h = 0; h < hkv; ++h) {
    codebook_consts(cb_K + 4 * h, host.data() + 16 * h);
    codebook_consts(cb_V + 4 * h, host.data() + 16 * h + 8);
  }
  for (int h = 0; h < hkv; ++h) {
    float* dst = const_cast<float*>(v.params) + (size_t)h * kParamFloats + kCbOff;
    if (cudaMemcpyAsync(dst, host.data() + 16 * h, 16 * sizeof(float), cudaMemcpyHostToDevice,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return OSCAR_ERR_CUDA;
  }
  return OSCAR_OK;
}

int oscar_set_rotation(oscar_cache* c, int layer, const float* U_K, const float* U_V, const float* tau_K,
                       const float* tau_V, void* stream) {
  if (!c || layer < 0 || layer >= c->lay.num_layers || !U_K || !tau_K || !tau_V) return OSCAR_ERR_INVALID_ARG;
  const bool expl = c->lay.v_mode == OSCAR_V_EXPLICIT;
  if (expl && !U_V) return OSCAR_ERR_INVALID_ARG;
  const int hkv = c->lay.num_kv_heads;
  for (int h = 0; h < hkv; ++h) {
    for (int which = 0; which < 2; ++which) {
      const float* U = which == 0 ? U_K : U_V;
      if (!U) continue;
      U += (size_t)h * kD * kD;
      for (int i = 0; i < kD; ++i)
        for (int j = i; j < kD; ++j) {
          double s = 0.0;
          for (int r = 0; r < kD; ++r) s += (double)U[r * kD + i] * (double)U[r * kD + j];
          const double e = std::fabs(s - (i == j ? 1.0 : 0.0));
          if (!(e <= 1e-3)) return OSCAR_ERR_NOT_ORTHOGONAL;
        }
    }
  }
  std::vector<float> host((size_t)hkv * kParamFloats, 0.f);
  for (int h = 0; h < hkv; ++h) {
    float* dst = host.data() + (size_t)h * kParamFloats;
    std::memcpy(dst + kUKOff, U_K + (size_t)h * kD * kD, kD * kD * sizeof(float));
    {
      const std::vector<double> R = composite_rotation(U_K + (size_t)h * kD * kD);
      rotation_fragments(R, reinterpret_cast<uint32_t*>(dst + kRKFragOff));
      rotation_image(R, reinterpret_cast<uint8_t*>(dst + kRKImgOff));
    }
    if (U_V) {
      const float* u = U_V + (size_t)h * kD * kD;
      std::memcpy(dst + kUVOff, u, kD * kD * sizeof(float));
      for (int i = 0; i < kD; ++i)
        for (int j = 0; j < kD; ++j) dst[kUVtOff + j * kD + i] = u[i * kD + j];
      if (expl) {
        const std::vector<double> R = composite_rotation(u);
        rotation_fragments(R, reinterpret_cast<uint32_t*>(dst + kRVFragOff));
        rotation_image(R, reinterpret_cast<uint8_t*>(dst + kRVImgOff));
      }
    }
    std::memcpy(dst + kTauKOff, tau_K + (size_t)h * kD, kD * sizeof(float));
    std::memcpy(dst + kTauVOff, tau_V + (size_t)h * kD, kD * sizeof(float));
    // compact-format grid per (kind, group): T = the group's largest threshold, D = fl32(2T / 255),
    // E = fl32(D / 3) (single-precision operations, each correctly rounded)
    for (int kind = 0; kind < 2; ++kind)
      for (int g = 0; g < kNG; ++g) {
        const float* t = (kind == 0 ? tau_K : tau_V) + (size_t)h * kD + g * kG;
        float T = t[0];
        for (int j = 1; j < kG; ++j) T = t[j] > T ? t[j] : T;
        const float D = (T + T) / 255.0f;
        const float E = D / 3.0f;
        float* mc = dst + kMetaCOff + kind * 8 + g * 4;
        mc[0] = T;
        mc[1] = D;
        mc[2] = E;
        mc[3] = 0.f;
      }
    static const uint8_t kUniform[4] = {0, 85, 170, 255};
    codebook_consts(kUniform, dst + kCbOff);
    codebook_consts(kUniform, dst + kCbOff + 8);
  }
  LayerView v = view(c, layer);
  cudaError_t e = cudaMemcpyAsync(const_cast<float*>(v.params), host.data(), host.size() * sizeof(float),
                                  cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
  // the source is pageable: the call returns once `host` has been staged, so it may be freed
  return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int oscar_quantize_prefill(oscar_cache* c, int layer, int B, const void* k, const void* v, const int32_t* cu_seqlens,
                           int total_tokens, const int32_t* hist_pt, int max_hist_pages, const int32_t* bf16_pt,
                           void* stream) {
  if (!c || layer < 0 || layer >= c->lay.num_layers || B < 0 || total_tokens < 0 || max_hist_pages < 0)
    return OSCAR_ERR_INVALID_ARG;
  if (B == 0 || total_tokens == 0) return OSCAR_OK;
  if (!k || !v || !cu_seqlens || !bf16_pt || (max_hist_pages > 0 && !hist_pt)) return OSCAR_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v)) return OSCAR_ERR_INVALID_ARG;
  return launch_prefill(view(c, layer), B, k, v, cu_seqlens, total_tokens, hist_pt, max_hist_pages, bf16_pt,
                        static_cast<cudaStream_t>(stream));
}

int oscar_project_quantize_prefill(oscar_cache* c, int layer, int B, const void* x, int d_model, const void* w_k,
                                   const void* w_v, const int32_t* cu_seqlens, int total_tokens,
                                   const int32_t* hist_pt, int max_hist_pages, const int32_t* bf16_pt, void* stream) {
  if (!c || layer < 0 || layer >= c->lay.num_layers || B < 0 || total_tokens < 0 || max_hist_pages < 0 ||
      d_model <= 0)
    return OSCAR_ERR_INVALID_ARG;
  if (B == 0 || total_tokens == 0) return OSCAR_OK;
  if (!x || !w_k || !w_v || !cu_seqlens || !bf16_pt || (max_hist_pages > 0 && !hist_pt)) return OSCAR_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_k) || !aligned16(w_v)) return OSCAR_ERR_INVALID_ARG;
  return launch_project_prefill(view(c, layer), B, x, d_model, w_k, w_v, cu_seqlens, total_tokens, hist_pt,
                                max_hist_pages, bf16_pt, static_cast<cudaStream_t>(stream));
}

int oscar_append_kv(oscar_cache* c, int layer, int B, const void* k, const void* v, const int32_t* seq_lens_before,
                    const int32_t* hist_pt, int max_hist_pages, const int32_t* bf16_pt, void* stream) {
  if (!c || layer < 0 || layer >= c->lay.num_layers || B < 0 || max_hist_pages < 0) return OSCAR_ERR_INVALID_ARG;
  if (B == 0) return OSCAR_OK;
  if (!k || !v || !seq_lens_before || !bf16_pt || (max_hist_pages > 0 && !hist_pt)) return OSCAR_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v)) return OSCAR_ERR_INVALID_ARG;
  return launch_prologue(view(c, layer), DecodeWorkspace{}, B, nullptr, k, v, seq_lens_before, hist_pt,
                         max_hist_pages, bf16_pt, 1.f, static_cast<cudaStream_t>(stream));
}

int oscar_set_decode_algo(oscar_cache* c, int algo) {
  if (!c || (algo != OSCAR_DECODE_SIMT && algo != OSCAR_DECODE_MMA && algo != OSCAR_DECODE_TC))
    return OSCAR_ERR_INVALID_ARG;
  c->algo = algo;
  return OSCAR_OK;
}

}  // extern "C"

namespace {

// Splits of a decode call: the request's own history pages (from shared_pages on) by the split
// policy, and on the tensor-core path the shared-prefix pages in one wave of CTAs (one per SM) over
// the kv heads and 128-row query tiles, within the max_splits slot budget.
void set_splits(const oscar_cache* c, int B, int max_hist_pages, int shared_pages, DecodeArgs& a) {
  const int hkv = c->lay.num_kv_heads, gq = c->lay.num_q_heads / c->lay.num_kv_heads;
  a.shared_pages = 0;
  a.nsplit_shared = 0;
  if (shared_pages > 0 && a.algo != OSCAR_DECODE_SIMT && c->lay.max_splits >= 2) {
    decode_split_policy(B, hkv, gq, a.nbf, max_hist_pages - shared_pages, c->lay.max_splits - 1, c->sms, a.algo,
                        &a.nsplit, &a.pages_per_split, &a.mma_occupancy);
    const int qtiles = (B * gq + kSharedRows - 1) / kSharedRows;
    int ns = std::max(1, c->sms / (hkv * qtiles));
    ns = std::min(std::min(ns, shared_pages), c->lay.max_splits - a.nsplit);
    a.shared_pages = shared_pages;
    a.nsplit_shared = ns;
    return;
  }
  decode_split_policy(B, hkv, gq, a.nbf, max_hist_pages, c->lay.max_splits, c->sms, a.algo, &a.nsplit,
                      &a.pages_per_split, &a.mma_occupancy);
}

int decode_impl(oscar_cache* c, int layer, int B, const void* q, const int32_t* seq_lens, const int32_t* hist_pt,
                int max_hist_pages, int shared_pages, const int32_t* bf16_pt, float sm_scale, void* out,
                int out_dtype, float* lse, void* stream) {
  if (!c || layer < 0 || layer >= c->lay.num_layers || B < 0 || B > c->lay.max_batch || max_hist_pages < 0)
    return OSCAR_ERR_INVALID_ARG;
  if (shared_pages < 0 || shared_pages > max_hist_pages) return OSCAR_ERR_INVALID_ARG;
  if (out_dtype != OSCAR_OUT_BF16 && out_dtype != OSCAR_OUT_FP32) return OSCAR_ERR_INVALID_ARG;
  if (B == 0) return OSCAR_OK;
  if (!q || !seq_lens || !bf16_pt || !out || (max_hist_pages > 0 && !hist_pt)) return OSCAR_ERR_INVALID_ARG;
  if (!aligned16(q)) return OSCAR_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return OSCAR_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
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
  a.algo = resolve_decode_algo(c->algo, c->lay.meta_format, c->lay.num_q_heads / c->lay.num_kv_heads);
  a.len_add = 0;
  a.skip_qprep = 0;
  a.nbf = (c->lay.sink + c->lay.recent) / kP;
  set_splits(c, B, max_hist_pages, shared_pages, a);
  a.ev0 = a.ev1 = nullptr;
  if (c->prof_on && c->prof_n < c->prof_cap) {
    a.ev0 = c->prof_ev[2 * c->prof_n];
    a.ev1 = c->prof_ev[2 * c->prof_n + 1];
    c->prof_n++;
  }
  return launch_decode(view(c, layer), c->dws, a, st);
}

int step_impl(oscar_cache* c, int layer, int B, const void* q, const void* k, const void* v,
              const int32_t* seq_lens_before, const int32_t* hist_pt, int max_hist_pages, int shared_pages,
              const int32_t* bf16_pt, float sm_scale, void* out, int out_dtype, float* lse, void* stream) {
  if (!c || layer < 0 || layer >= c->lay.num_layers || B < 0 || B > c->lay.max_batch || max_hist_pages < 0)
    return OSCAR_ERR_INVALID_ARG;
  if (shared_pages < 0 || shared_pages > max_hist_pages) return OSCAR_ERR_INVALID_ARG;
  if (out_dtype != OSCAR_OUT_BF16 && out_dtype != OSCAR_OUT_FP32) return OSCAR_ERR_INVALID_ARG;
  if (B == 0) return OSCAR_OK;
  if (!q || !k || !v || !seq_lens_before || !bf16_pt || !out || (max_hist_pages > 0 && !hist_pt))
    return OSCAR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return OSCAR_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return OSCAR_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LayerView lv = view(c, layer);
  DecodeArgs a;
  a.B = B;
  a.q = q;
  a.seq_lens = seq_lens_before;
  a.len_add = 1;                         // attend over the appended token too
  a.skip_qprep = 1;                      // the step prologue below rotates the queries
  a.hist_pt = hist_pt;
  a.max_hist_pages = max_hist_pages;
  a.bf16_pt = bf16_pt;
  a.sm_scale = sm_scale;
  a.out = out;
  a.out_dtype = out_dtype;
  a.lse = lse;
  a.algo = resolve_decode_algo(c->algo, c->lay.meta_format, c->lay.num_q_heads / c->lay.num_kv_heads);
  a.nbf = (c->lay.sink + c->lay.recent) / kP;
  set_splits(c, B, max_hist_pages, shared_pages, a);
  a.ev0 = a.ev1 = nullptr;
  if (c->prof_on && c->prof_n < c->prof_cap) {
    a.ev0 = c->prof_ev[2 * c->prof_n];
    a.ev1 = c->prof_ev[2 * c->prof_n + 1];
    c->prof_n++;
  }
  // one prologue launch (append with demotion, and the query prologue), then the decode and the
  // merge, each a programmatic dependent of the kernel before it
  const int rc = launch_prologue(lv, c->dws, B, q, k, v, seq_lens_before, hist_pt, max_hist_pages, bf16_pt,
                                 sm_scale, st);
  if (rc != OSCAR_OK) return rc;
  return launch_decode(lv, c->dws, a, st);
}

}  // namespace

extern "C" {

int oscar_decode_attention(oscar_cache* c, int layer, int B, const void* q, const int32_t* seq_lens,
                           const int32_t* hist_pt, int max_hist_pages, const int32_t* bf16_pt, float sm_scale,
                           void* out, int out_dtype, float* lse, void* stream) {
  return decode_impl(c, layer, B, q, seq_lens, hist_pt, max_hist_pages, 0, bf16_pt, sm_scale, out, out_dtype, lse,
                     stream);
}

int oscar_decode_attention_shared(oscar_cache* c, int layer, int B, const void* q, const int32_t* seq_lens,
                                  const int32_t* hist_pt, int max_hist_pages, int shared_hist_pages,
                                  const int32_t* bf16_pt, float sm_scale, void* out, int out_dtype, float* lse,
                                  void* stream) {
  return decode_impl(c, layer, B, q, seq_lens, hist_pt, max_hist_pages, shared_hist_pages, bf16_pt, sm_scale, out,
                     out_dtype, lse, stream);
}

int oscar_decode_step(oscar_cache* c, int layer, int B, const void* q, const void* k, const void* v,
                      const int32_t* seq_lens_before, const int32_t* hist_pt, int max_hist_pages,
                      const int32_t* bf16_pt, float sm_scale, void* out, int out_dtype, float* lse, void* stream) {
  return step_impl(c, layer, B, q, k, v, seq_lens_before, hist_pt, max_hist_pages, 0, bf16_pt, sm_scale, out,
                   out_dtype, lse, stream);
}

int oscar_decode_step_shared(oscar_cache* c, int layer, int B, const void* q, const void* k, const void* v,
                             const int32_t* seq_lens_before, const int32_t* hist_pt, int max_hist_pages,
                             int shared_hist_pages, const int32_t* bf16_pt, float sm_scale, void* out, int out_dtype,
                             float* lse, void* stream) {
  return step_impl(c, layer, B, q, k, v, seq_lens_before, hist_pt, max_hist_pages, shared_hist_pages, bf16_pt,
                   sm_scale, out, out_dtype, lse, stream);
}

int oscar_get_status(oscar_cache* c, int* code) {
  if (!c || !code) return OSCAR_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return OSCAR_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, c->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return OSCAR_ERR_CUDA;
  if (cudaMemset(c->status, 0, sizeof(int)) != cudaSuccess) return OSCAR_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return OSCAR_ERR_CUDA;
  *code = v;
  return v == 0 ? OSCAR_OK : OSCAR_ERR_DEVICE_STATUS;
}

int oscar_pack_rotated(oscar_cache* c, int layer, int kind, const float* xrot, const int32_t* page_ids,
                       const int32_t* rows, int N, void* stream) {
  if (!c || layer < 0 || layer >= c->lay.num_layers || N < 0 || (kind != OSCAR_KIND_K && kind != OSCAR_KIND_V))
    return OSCAR_ERR_INVALID_ARG;
  if (N == 0) return OSCAR_OK;
  if (!xrot || !page_ids || !rows) return OSCAR_ERR_INVALID_ARG;
  return launch_pack_rotated(view(c, layer), kind, xrot, page_ids, rows, N, static_cast<cudaStream_t>(stream));
}

int oscar_rotate(oscar_cache* c, int layer, int kind, const void* x, float* y, int N, void* stream) {
  if (!c || layer < 0 || layer >= c->lay.num_layers || N < 0 || (kind != OSCAR_KIND_K && kind != OSCAR_KIND_V))
    return OSCAR_ERR_INVALID_ARG;
  if (N == 0) return OSCAR_OK;
  if (!x || !y) return OSCAR_ERR_INVALID_ARG;
  return launch_rotate(view(c, layer), kind, x, y, N, static_cast<cudaStream_t>(stream));
}

int oscar_bf16_decode_workspace_bytes(int max_batch, int num_q_heads, int max_splits, size_t* bytes) {
  if (max_batch < 1 || num_q_heads < 1 || max_splits < 1 || !bytes) return OSCAR_ERR_INVALID_ARG;
  *bytes = kAlign + align_up((size_t)max_batch * num_q_heads * max_splits * kPartFloats * sizeof(float));
  return OSCAR_OK;
}

int oscar_bf16_decode(int B, int num_q_heads, int num_kv_heads, const void* kv_pages, int num_pages, const void* q,
                      const int32_t* seq_lens, const int32_t* page_table, int max_pages, float sm_scale, void* out,
                      int out_dtype, float* lse, void* workspace, size_t workspace_bytes, int max_splits,
                      void* stream) {
  if (B < 0 || num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads || num_pages < 0 || max_pages < 1 ||
      max_splits < 1)
    return OSCAR_ERR_INVALID_ARG;
  if (!is_pow2_le8(num_q_heads / num_kv_heads)) return OSCAR_ERR_UNSUPPORTED;
  if (out_dtype != OSCAR_OUT_BF16 && out_dtype != OSCAR_OUT_FP32) return OSCAR_ERR_INVALID_ARG;
  if (B == 0) return OSCAR_OK;
  if (!kv_pages || !q || !seq_lens || !page_table || !out || !workspace) return OSCAR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return OSCAR_ERR_INVALID_ARG;
  size_t need = 0;
  oscar_bf16_decode_workspace_bytes(B, num_q_heads, max_splits, &need);
  if (workspace_bytes < need) return OSCAR_ERR_INVALID_ARG;
  int rc = configure_once();
  if (rc != OSCAR_OK) return rc;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OSCAR_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return OSCAR_ERR_CUDA;
  // the streaming kernel holds two CTAs per SM: one wave of splits over the (request, kv head) pairs
  const long units = (long)B * num_kv_heads;
  int nsplit = (int)std::max(1L, 2L * sms / units);
  nsplit = std::min(std::min(nsplit, max_splits), max_pages);
  const int pps = (max_pages + nsplit - 1) / nsplit;
  nsplit = (max_pages + pps - 1) / pps;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  return launch_bf16_decode(B, num_q_heads, num_kv_heads, kv_pages, num_pages, q, seq_lens, page_table, max_pages,
                            sm_scale, out, out_dtype, lse, reinterpret_cast<float*>(w + kAlign), max_splits, nsplit,
                            pps, reinterpret_cast<int*>(w), static_cast<cudaStream_t>(stream));
}

int oscar_trace_ctas(oscar_cache* c, void* buf, int capacity) {
  if (!c || capacity < 0 || (buf != nullptr && capacity == 0)) return OSCAR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(buf) % 8) return OSCAR_ERR_INVALID_ARG;
  c->dws.cta_trace = static_cast<unsigned long long*>(buf);
  c->dws.trace_cap = buf ? capacity : 0;
  return OSCAR_OK;
}

int oscar_check_wait_timeout(oscar_cache* c, void* stream) {
  if (!c) return OSCAR_ERR_INVALID_ARG;
  return launch_wait_probe(c->status, static_cast<cudaStream_t>(stream));
}

int oscar_trace_timeline(oscar_cache* c, void* buf, int capacity) {
  if (!c || capacity < 0 || (buf != nullptr && capacity == 0)) return OSCAR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(buf) % 8) return OSCAR_ERR_INVALID_ARG;
  c->timeline = static_cast<unsigned long long*>(buf);
  c->timeline_cap = buf ? capacity : 0;
  return OSCAR_OK;
}

int oscar_profile_begin(oscar_cache* c, int capacity) {
  if (!c || capacity < 1) return OSCAR_ERR_INVALID_ARG;
  while ((int)c->prof_ev.size() < 2 * capacity) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return OSCAR_ERR_CUDA;
    c->prof_ev.push_back(e);
  }
  c->prof_cap = capacity;
  c->prof_n = 0;
  c->prof_on = true;
  return OSCAR_OK;
}

int oscar_profile_read(oscar_cache* c, double* total_ms, int* launches) {
  if (!c || !total_ms || !launches) return OSCAR_ERR_INVALID_ARG;
  c->prof_on = false;
  double tot = 0.0;
  for (int i = 0; i < c->prof_n; ++i) {
    if (cudaEventSynchronize(c->prof_ev[2 * i + 1]) != cudaSuccess) return OSCAR_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, c->prof_ev[2 * i], c->prof_ev[2 * i + 1]) != cudaSuccess) return OSCAR_ERR_CUDA;
    tot += ms;
  }
  *total_ms = tot;
  *launches = c->prof_n;
  return OSCAR_OK;
}

}  // extern "C"

namespace oscar {

// Device view of layer `layer` of a pool laid out for `L`, with its status
// word at `status`; for entry points that work without a cache handle.
int pool_layer_view(const oscar_layout* L, void* pool, int layer, int* status, LayerView* out) {
  int rc = check_layout(L);
  if (rc != OSCAR_OK) return rc;
  if (!pool || !out || layer < 0 || layer >= L->num_layers) return OSCAR_ERR_INVALID_ARG;
  size_t int2b, bf16b, prmb, layerb, poolb, wsb;
  sizes(L, &int2b, &bf16b, &prmb, &layerb, &poolb, &wsb);
  uint8_t* base = static_cast<uint8_t*>(pool) + (size_t)layer * layerb;
  out->int2 = base;
  out->bf16 = base + int2b;
  out->params = reinterpret_cast<const float*>(base + int2b + bf16b);
  out->next_params = nullptr;
  out->n_int2 = L->num_int2_pages;
  out->n_bf16 = L->num_bf16_pages;
  out->hkv = L->num_kv_heads;
  out->hq = L->num_q_heads;
  out->sink = L->sink;
  out->recent = L->recent;
  out->v_explicit = L->v_mode == OSCAR_V_EXPLICIT;
  out->meta_u8 = L->meta_format == OSCAR_META_U8;
  out->meta_cb = L->meta_format == OSCAR_META_CB;
  out->blk_bytes = out->meta_u8 ? kBlockBytesU8 : kBlockBytes;
  out->status = status;
  out->layer = layer;
  out->timeline = nullptr;
  out->timeline_cap = 0;
  return OSCAR_OK;
}

// The history split choice of oscar_decode_attention, for at most max_splits splits.
void decode_split_policy(int B, int hkv, int gq, int nbf, int max_pages, int max_splits, int sms, int algo,
                         int* nsplit, int* pps, int* occupancy) {
  *occupancy = 3;
  if (algo == OSCAR_DECODE_TC) choose_splits_tc(B, hkv, max_pages, max_splits, sms, nsplit, pps);
  else if (algo == OSCAR_DECODE_MMA) choose_splits_mma(B, hkv, gq, nbf, max_pages, max_splits, sms, nsplit, pps, occupancy);
  else choose_splits_simt(B, hkv, max_pages, max_splits, sms, nsplit, pps);
}

int configure_kernels() { return configure_once(); }

}  // namespace oscar
