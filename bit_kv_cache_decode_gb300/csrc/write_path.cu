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
  quantize_pack_row(y, tau, int2_block_w(lv, page, h), row, kind, lv.meta_u8 ? meta_consts(lv, h, kind) : nullptr,
                    lv.meta_cb ? cb_consts(lv, h, kind) : nullptr, lv.status);
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

int configure_write_path_kernels() {
  if (configure_prefill_kernel() != OSCAR_OK) return OSCAR_ERR_CUDA;
  if (configure_project_prefill_kernel() != OSCAR_OK) return OSCAR_ERR_CUDA;
  if (configure_prologue_kernel() != OSCAR_OK) return OSCAR_ERR_CUDA;
  return OSCAR_OK;
}

}  // namespace oscar
