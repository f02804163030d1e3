// Step prologue (sm_103a): the append with demotion and the decode's query
// prologue in one launch.
//
// * Append (news article "超越 TurboQuant…OSCAR…", section "OSCAR 的设计思路":
//   the new token enters the recent window, and the oldest recent token is
//   rotated, clipped, quantised and packed into the history).
// * Query prologue (MarkTechPost article "Together AI 开源 OSCAR…", section
//   "OSCAR 有何不同做法": R_K = U_Q H_Had P_br; the read path's inverse rotation
//   of the keys is applied once to the query instead, R_K being orthogonal).
//
// grid = (B, hkv, 2 kinds or 1), block = 256 (8 warps). CTA (b, h, kind):
// * The demoted row of this kind (if the recent window is full) is row 0 of a
//   16-row tile. For kind K with queries, the gq query rows of kv head h are
//   rows 1 .. gq.
// * One tensor-core pass multiplies the tile by the composite rotation (R_K, or
//   R_V in explicit-V mode; V in V-absorbed mode is not rotated). Its fragments
//   come from the rotation parameters in 8 bulk copies.
// * The last warp quantises and packs the demoted row (the same single-row quantiser
//   as everywhere) into its history row.
// * The query rows become q~, its group sums, scale factors and the MMA
//   fragments of the tensor-core decode (qprep.cuh).
// * The new token is written to its ring slot, after the slot's old row was
//   staged.
// The grid waits for the kernel before it on the stream (programmatic
// dependent launch) before it reads q, k and v, then lets the decode be
// scheduled. Sequence lengths, page tables and the pool's rows (inputs the
// kernel before does not produce) are read before that wait.
#include "kernels.cuh"
#include "rotate.cuh"
#include "tma.cuh"
#include "timeline.cuh"
#include "qprep.cuh"

namespace oscar {
namespace {

__device__ __forceinline__ bool valid_page(int p, int n) { return p >= 0 && p < n; }

// smem: rotation fragments | 16-row tile | tau | 8 mbarriers
constexpr int kTileFloats = 16 * kTileStride;

__global__ void __launch_bounds__(kPrologueWarps * 32, 1)
    k_step_prologue(LayerView lv, DecodeWorkspace ws, const __nv_bfloat16* __restrict__ q,
                    const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                    const int* __restrict__ seq_lens_before, const int* __restrict__ hist_pt, int max_hist_pages,
                    const int* __restrict__ bf16_pt, float scale_log2) {
  TimelineSpan timeline_span(lv, k != nullptr ? kTlAppend : kTlQprep);
  extern __shared__ __align__(128) float smem[];
  uint32_t* frag_s = reinterpret_cast<uint32_t*>(smem);
  float* rows = smem + kRFragWords;                  // [16][kTileStride]
  float* tau_s = rows + kTileFloats;                 // [128]
  const uint32_t bars = smem_addr(tau_s + kD);
  __shared__ int sig[8];
  const int b = blockIdx.x, h = blockIdx.y, kind = blockIdx.z;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int gq = lv.hq / lv.hkv;
  const float* prm = lv.params + (size_t)h * kParamFloats;
  const bool do_q = q != nullptr && kind == OSCAR_KIND_K;
  const bool rotate = (kind == OSCAR_KIND_K) || lv.v_explicit;
  // The rotation fragments do not depend on the kernel before: they are requested before the wait below,
  // while that kernel still runs (this grid is scheduled early). Every CTA that may rotate requests them.
  const bool fetch_frags = rotate && (do_q || k != nullptr);
  if (fetch_frags && tid == 0) {
    const float* f = prm + (kind == OSCAR_KIND_K ? kRKFragOff : kRVFragOff);
    const uint64_t keep = l2_evict_last();
    constexpr int chunk = kRFragWords / 8;             // one k-block: 2,048 words
    for (int c = 0; c < 8; ++c) {
      mbar_init(bars + 8 * c);
      bulk_load_hint(smem_addr(frag_s + c * chunk), f + c * chunk, chunk * 4, bars + 8 * c, keep);
    }
  }
  // --- demotion of the oldest recent token: where it comes from and goes to ---
  // Sequence lengths, page tables and the pool are not produced by the kernel before this one (the
  // caller's q, k, v are): they are read before the programmatic wait, so only q, k and v wait for it.
  const int bf16_per_req = (lv.sink + lv.recent) / kP;
  int L_old = 0;
  bool demote = false;
  int slot = 0, spage = -1, hh = 0, hpage = -1;
  if (k != nullptr) {
    L_old = __ldcg(seq_lens_before + b);          // L2 reads: nothing older may sit in this SM's L1
    if (L_old < 0 && tid == 0) flag(lv.status, OSCAR_STATUS_BAD_SEQLEN);
    demote = L_old >= lv.sink + lv.recent;
    if (demote) {
      const int old = L_old - lv.recent;
      slot = (old - lv.sink) % lv.recent;
      spage = __ldcg(bf16_pt + b * bf16_per_req + lv.sink / kP + slot / kP);
      hh = old - lv.sink;
      const bool ok_h = hh / kP < max_hist_pages;
      hpage = ok_h ? __ldcg(hist_pt + (size_t)b * max_hist_pages + hh / kP) : -1;
      if (!ok_h || !valid_page(spage, lv.n_bf16) || !valid_page(hpage, lv.n_int2)) {
        if (tid == 0) flag(lv.status, ok_h ? OSCAR_STATUS_BAD_PAGE : OSCAR_STATUS_BAD_SEQLEN);
        demote = false;
      }
    }
  }
  // The next layer's prologue needs its rotation fragments from L2 about one layer's decode from now:
  // ask for them now, with the same evict-last priority, so the page stream of this layer does not
  // leave them to be fetched from HBM on the next critical path.
  if (lv.next_params != nullptr && b == 0 && tid == 0 && rotate) {
    const float* nf = lv.next_params + (size_t)h * kParamFloats + (kind == OSCAR_KIND_K ? kRKFragOff : kRVFragOff);
    l2_prefetch(nf, kRFragWords * 4, l2_evict_last());
  }
  const bool need_frags = (demote && rotate) || do_q;      // fetch_frags holds whenever this does
  // --- the tile: row 0 the demoted row, rows 1 .. gq the queries, zeros elsewhere ---
  // one 16-byte chunk (8 values) per thread: 16 rows x 16 chunks; the demoted row's chunks are loaded
  // before the wait, the queries' after it
  static_assert(kPrologueWarps * 32 == 16 * 16, "one chunk per thread");
  const int r = tid >> 4, c8 = tid & 15;
  uint4 u = make_uint4(0u, 0u, 0u, 0u);
  if (r == 0 && demote) u = __ldcg(reinterpret_cast<const uint4*>(bf16_row(lv, spage, h, kind, slot % kP) + 8 * c8));
  // Wait for the grid before (in a model, the kernel that made q, k and v), then let the decode be
  // scheduled; it waits for this grid before it reads anything this kernel writes.
  pdl_wait();
  pdl_launch_dependents();
  if (r >= 1 && r <= gq && do_q) {
    u = *reinterpret_cast<const uint4*>(q + ((size_t)b * lv.hq + h * gq + r - 1) * kD + 8 * c8);
    if (bf16x2_nonfinite(u.x) || bf16x2_nonfinite(u.y) || bf16x2_nonfinite(u.z) || bf16x2_nonfinite(u.w))
      flag(lv.status, OSCAR_STATUS_NONFINITE);
  }
  {
    const uint32_t wds[4] = {u.x, u.y, u.z, u.w};
    float4* dst = reinterpret_cast<float4*>(rows + r * kTileStride + 8 * c8);
    dst[0] = make_float4(__uint_as_float(wds[0] << 16), __uint_as_float(wds[0] & 0xffff0000u),
                         __uint_as_float(wds[1] << 16), __uint_as_float(wds[1] & 0xffff0000u));
    dst[1] = make_float4(__uint_as_float(wds[2] << 16), __uint_as_float(wds[2] & 0xffff0000u),
                         __uint_as_float(wds[3] << 16), __uint_as_float(wds[3] & 0xffff0000u));
  }
  if (tid < kD) tau_s[tid] = prm[(kind == OSCAR_KIND_K ? kTauKOff : kTauVOff) + tid];
  __syncthreads();                                   // barriers initialised, tile staged, old slot read
  if (need_frags && !rotate_tile16(frag_s, rows, bars)) {
    if (tid == 0) flag(lv.status, OSCAR_STATUS_TIMEOUT);
    mbar_wait(bars + 8 * w, 0);                      // one more bounded wait for the copies in flight
    return;                                          // the pool is left untouched
  }
  if (fetch_frags && !need_frags) mbar_wait(bars + 8 * w, 0);   // copies requested but unused: let them land
  timeline_span.mark();                              // rotation done (fragments and rows loaded)
  // rows now hold rotated values in rotated channel order (row 0 raw if V is not rotated). The last
  // warp quantises the demoted row while warps 0 .. 6 finish the queries (named barrier 1).
  if (w == kPrologueWarps - 1) {
    if (demote) {
      float y[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) y[r] = rows[rot_channel(lane, r)];
      quantize_pack_row(y, tau_s, int2_block_w(lv, hpage, h), hh % kP, kind,
                        lv.meta_u8 ? meta_consts(lv, h, kind) : nullptr, lv.meta_cb ? cb_consts(lv, h, kind) : nullptr,
                        lv.status);
    }
  } else if (do_q) {
    constexpr int kQWarps = kPrologueWarps - 1;
    qprep_stats(lv, ws, rows + kTileStride, kTileStride, sig, b, h, kQWarps);
    asm volatile("bar.sync 1, %0;" ::"n"(kQWarps * 32) : "memory");
    qprep_finish(lv, ws, rows + kTileStride, kTileStride, sig, b, h, scale_log2, kQWarps);
  }
  // --- the new token into its slot (the old row was staged before the first barrier) ---
  if (k == nullptr || L_old < 0 || w != kPrologueWarps - 2) return;
  const int pos = L_old;
  int page, row;
  if (pos < lv.sink) {
    page = bf16_pt[b * bf16_per_req + pos / kP];
    row = pos % kP;
  } else {
    const int s2 = (pos - lv.sink) % lv.recent;
    page = bf16_pt[b * bf16_per_req + lv.sink / kP + s2 / kP];
    row = s2 % kP;
  }
  if (!valid_page(page, lv.n_bf16)) {
    if (lane == 0) flag(lv.status, OSCAR_STATUS_BAD_PAGE);
    return;
  }
  const __nv_bfloat16* src = (kind == OSCAR_KIND_K ? k : v) + ((size_t)b * lv.hkv + h) * kD;
  const uint2 x = reinterpret_cast<const uint2*>(src)[lane];
  if (__any_sync(0xffffffffu, bf16x2_nonfinite(x.x) || bf16x2_nonfinite(x.y)) && lane == 0)
    flag(lv.status, OSCAR_STATUS_NONFINITE);
  reinterpret_cast<uint2*>(bf16_row(lv, page, h, kind, row))[lane] = x;
}

constexpr int kPrologueSmem = (kRFragWords + kTileFloats + kD) * 4 + 64;

}  // namespace

int launch_prologue(const LayerView& lv, const DecodeWorkspace& ws, int B, const void* q, const void* k,
                    const void* v, const int* seq_lens_before, const int* hist_pt, int max_hist_pages,
                    const int* bf16_pt, float sm_scale, cudaStream_t st) {
  if (B == 0) return OSCAR_OK;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(B, lv.hkv, k != nullptr ? 2 : 1);   // query-only: the K CTAs
  cfg.blockDim = dim3(kPrologueWarps * 32);
  cfg.dynamicSmemBytes = kPrologueSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_step_prologue, lv, ws, static_cast<const __nv_bfloat16*>(q),
                            static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v),
                            seq_lens_before, hist_pt, max_hist_pages, bf16_pt, sm_scale * kLog2e) == cudaSuccess
             ? OSCAR_OK
             : OSCAR_ERR_CUDA;
}

int configure_prologue_kernel() {
  if (cudaFuncSetAttribute(k_step_prologue, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrologueSmem) !=
      cudaSuccess)
    return OSCAR_ERR_CUDA;
  return set_max_shared_carveout(reinterpret_cast<const void*>(k_step_prologue));
}

}  // namespace oscar
