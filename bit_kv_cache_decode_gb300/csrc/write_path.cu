// Write path of the OSCAR mixed-precision token pool (sm_103a): rotate, clip,
// quantise, pack and place tokens (MarkTechPost article "Together AI 开源 OSCAR…",
// section "服务系统：混合精度缓存布局", write path; news article "超越 TurboQuant…
// OSCAR…", section "OSCAR 的设计思路": new tokens enter the recent window and the
// oldest recent token is demoted into the INT2 history).
#include "kernels.cuh"
#include "rotate.cuh"
#include "tma.cuh"
#include "timeline.cuh"

namespace oscar {

namespace {

__device__ __forceinline__ bool valid_page(int p, int n) { return p >= 0 && p < n; }

// Copy one bf16 row (128 values) from global to the float array xs (shared), one warp.
__device__ __forceinline__ void load_row_f32(const __nv_bfloat16* src, float* xs) {
  const int lane = threadIdx.x & 31;
  const __nv_bfloat162* s2 = reinterpret_cast<const __nv_bfloat162*>(src);
  float2 a = __bfloat1622float2(s2[lane]);
  float2 b = __bfloat1622float2(s2[lane + 32]);
  xs[2 * lane] = a.x; xs[2 * lane + 1] = a.y;
  xs[64 + 2 * lane] = b.x; xs[64 + 2 * lane + 1] = b.y;
}

// Copy one bf16 row (256 bytes) src -> dst, one warp (8 bytes per lane).
__device__ __forceinline__ void copy_row_bf16(const __nv_bfloat16* src, __nv_bfloat16* dst) {
  const int lane = threadIdx.x & 31;
  reinterpret_cast<uint2*>(dst)[lane] = reinterpret_cast<const uint2*>(src)[lane];
}

}  // namespace

// ---------------------------------------------------------------------------
// Pre-rotated float32 rows -> quantised INT2 history rows (debug / bit-exact check).
// One warp per (token, kv head).
__global__ void k_pack_rotated(LayerView lv, int kind, const float* __restrict__ xrot,
                               const int* __restrict__ page_ids, const int* __restrict__ rows, int N) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= N * lv.hkv) return;
  const int n = warp / lv.hkv, h = warp % lv.hkv;
  const int page = page_ids[n], row = rows[n];
  if (!valid_page(page, lv.n_int2) || row < 0 || row >= kP) {
    if (lane == 0) flag(lv.status, OSCAR_STATUS_BAD_PAGE);
    return;
  }
  const float* x = xrot + ((size_t)n * lv.hkv + h) * kD;
  float y[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) y[r] = x[rot_channel(lane, r)];
  const float* tau = lv.params + (size_t)h * kParamFloats + (kind == OSCAR_KIND_K ? kTauKOff : kTauVOff);
  quantize_pack_row(y, tau, int2_block_w(lv, page, h), row, kind);
}

// ---------------------------------------------------------------------------
// y = x R for N rows of every kv head (debug). One warp per (token, head).
__global__ void k_rotate(LayerView lv, int kind, const __nv_bfloat16* __restrict__ x, float* __restrict__ y, int N) {
  __shared__ float xs[4][kD];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int warp = blockIdx.x * (blockDim.x >> 5) + wib;
  if (warp >= N * lv.hkv) return;
  const int n = warp / lv.hkv, h = warp % lv.hkv;
  load_row_f32(x + ((size_t)n * lv.hkv + h) * kD, xs[wib]);
  __syncwarp();
  const float* U = lv.params + (size_t)h * kParamFloats + (kind == OSCAR_KIND_K ? kUKOff : kUVOff);
  float v[1][4];
  warp_rotate<1>(U, xs[wib], v);
  float* out = y + ((size_t)n * lv.hkv + h) * kD;
#pragma unroll
  for (int r = 0; r < 4; ++r) out[rot_channel(lane, r)] = v[0][r];
}

// ---------------------------------------------------------------------------
// Append one token per request with demotion. grid = (B, hkv, 2 kinds); block = 128.
// The CTA stages U in shared memory by one bulk copy (when a demotion needs
// it), rotates the demoted row with 4 warps each summing 32 rows of U, then
// warp 0 finishes the Hadamard/bit-reversal, quantises and packs. Only after
// that is the ring slot overwritten with the new token.
__global__ void __launch_bounds__(128) k_append(LayerView lv, const __nv_bfloat16* __restrict__ k,
                                                const __nv_bfloat16* __restrict__ v,
                                                const int* __restrict__ seq_lens_before,
                                                const int* __restrict__ hist_pt, int max_hist_pages,
                                                const int* __restrict__ bf16_pt) {
  TimelineSpan timeline_span(lv, kTlAppend);
  extern __shared__ __align__(128) float smem[];
  float* Us = smem;                 // [128][128]
  float* xs = smem + kD * kD;       // [128] demoted row
  float* part = xs + kD;            // [4][128]
  const uint32_t bar = smem_addr(part + 4 * kD);
  __shared__ int landed;
  const int b = blockIdx.x, h = blockIdx.y, kind = blockIdx.z;
  const int tid = threadIdx.x, wib = tid >> 5, lane = tid & 31;
  pdl_launch_dependents();          // the next kernel may start its prologue; it waits for this grid
  const int bf16_per_req = (lv.sink + lv.recent) / kP;
  const int L_old = seq_lens_before[b];
  const bool bad = L_old < 0;
  if (bad && tid == 0) flag(lv.status, OSCAR_STATUS_BAD_SEQLEN);
  const float* prm = lv.params + (size_t)h * kParamFloats;
  const bool rotate = (kind == OSCAR_KIND_K) || lv.v_explicit;
  // --- demotion of the oldest recent token: where it comes from and goes to ---
  bool demote = !bad && L_old >= lv.sink + lv.recent;
  int slot = 0, spage = -1, hh = 0, hpage = -1;
  if (demote) {
    const int old = L_old - lv.recent;
    slot = (old - lv.sink) % lv.recent;
    spage = bf16_pt[b * bf16_per_req + lv.sink / kP + slot / kP];
    hh = old - lv.sink;
    const bool ok_h = hh / kP < max_hist_pages;
    hpage = ok_h ? hist_pt[b * max_hist_pages + hh / kP] : -1;
    if (!ok_h || !valid_page(spage, lv.n_bf16) || !valid_page(hpage, lv.n_int2)) {
      if (tid == 0) flag(lv.status, ok_h ? OSCAR_STATUS_BAD_PAGE : OSCAR_STATUS_BAD_SEQLEN);
      demote = false;
    }
  }
  const bool need_u = demote && rotate;
  if (need_u && tid == 0) {
    mbar_init(bar);
    bulk_load_hint(smem_addr(Us), prm + (kind == OSCAR_KIND_K ? kUKOff : kUVOff), kD * kD * 4, bar, l2_evict_last());
  }
  if (demote && tid < 64) {
    const __nv_bfloat16* src = bf16_row(lv, spage, h, kind, slot % kP);
    float2 f = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(src)[tid]);
    xs[2 * tid] = f.x; xs[2 * tid + 1] = f.y;
  }
  if (tid == 0) landed = 1;
  __syncthreads();
  if (need_u && !mbar_wait(bar, 0)) landed = 0;
  __syncthreads();
  if (!landed) {                    // U never arrived: report, leave the pool untouched
    if (tid == 0) flag(lv.status, OSCAR_STATUS_TIMEOUT);
    return;
  }
  if (demote) {
    float y[4];
    if (rotate) {
      // warp w sums rows [32w, 32w+32) of U
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
      for (int i = wib * 32; i < wib * 32 + 32; ++i) {
        const float xi = xs[i];
        const float* row = Us + i * kD + lane;
        acc[0] = fmaf(xi, row[0], acc[0]); acc[1] = fmaf(xi, row[32], acc[1]);
        acc[2] = fmaf(xi, row[64], acc[2]); acc[3] = fmaf(xi, row[96], acc[3]);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) part[wib * kD + lane + 32 * r] = acc[r];
      __syncthreads();
      if (wib == 0) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int j = lane + 32 * r;
          y[r] = ((part[j] + part[kD + j]) + part[2 * kD + j]) + part[3 * kD + j];
        }
        fwht128(y);
      }
    } else if (wib == 0) {
#pragma unroll
      for (int r = 0; r < 4; ++r) y[r] = xs[rot_channel(lane, r)];
    }
    if (wib == 0) {
      const float* tau = prm + (kind == OSCAR_KIND_K ? kTauKOff : kTauVOff);
      quantize_pack_row(y, tau, int2_block_w(lv, hpage, h), hh % kP, kind);
    }
    __syncthreads();   // the slot is read above before it is overwritten below
  }
  // --- write the new token ---
  if (bad || wib != 0) return;
  const int pos = L_old;
  int page, row;
  if (pos < lv.sink) {
    page = bf16_pt[b * bf16_per_req + pos / kP]; row = pos % kP;
  } else {
    const int s2 = (pos - lv.sink) % lv.recent;
    page = bf16_pt[b * bf16_per_req + lv.sink / kP + s2 / kP]; row = s2 % kP;
  }
  if (!valid_page(page, lv.n_bf16)) { if (lane == 0) flag(lv.status, OSCAR_STATUS_BAD_PAGE); return; }
  const __nv_bfloat16* src = (kind == OSCAR_KIND_K ? k : v) + ((size_t)b * lv.hkv + h) * kD;
  copy_row_bf16(src, bf16_row(lv, page, h, kind, row));
}

// ---------------------------------------------------------------------------
// host launchers

int launch_pack_rotated(const LayerView& lv, int kind, const float* xrot, const int* page_ids, const int* rows,
                        int N, cudaStream_t st) {
  if (N == 0) return OSCAR_OK;
  const int warps = N * lv.hkv, wpb = 4;
  k_pack_rotated<<<(warps + wpb - 1) / wpb, wpb * 32, 0, st>>>(lv, kind, xrot, page_ids, rows, N);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int launch_rotate(const LayerView& lv, int kind, const void* x, float* y, int N, cudaStream_t st) {
  if (N == 0) return OSCAR_OK;
  const int warps = N * lv.hkv, wpb = 4;
  k_rotate<<<(warps + wpb - 1) / wpb, wpb * 32, 0, st>>>(lv, kind, static_cast<const __nv_bfloat16*>(x), y, N);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int launch_append(const LayerView& lv, int B, const void* k, const void* v, const int* seq_lens_before,
                  const int* hist_pt, int max_hist_pages, const int* bf16_pt, cudaStream_t st) {
  if (B == 0) return OSCAR_OK;
  dim3 grid(B, lv.hkv, 2);
  k_append<<<grid, 128, kAppendSmem, st>>>(lv, static_cast<const __nv_bfloat16*>(k),
                                           static_cast<const __nv_bfloat16*>(v), seq_lens_before, hist_pt,
                                           max_hist_pages, bf16_pt);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int configure_write_path_kernels() {
  if (configure_prefill_kernel() != OSCAR_OK) return OSCAR_ERR_CUDA;
  if (cudaFuncSetAttribute(k_append, cudaFuncAttributeMaxDynamicSharedMemorySize, kAppendSmem) != cudaSuccess)
    return OSCAR_ERR_CUDA;
  return OSCAR_OK;
}

}  // namespace oscar
