// Log-sum-exp merge of a decode call's partial results (sm_103a), shared by
// both decode algorithms (the online-softmax merge of split partials: Page A of
// the OSCAR write-ups, "online softmax"; partial = (m, l, acc) with l and acc
// relative to 2^m, m in log2 units).
//
// grid = (Hq, B), block = 256: one CTA per (request, query head). The head's
// slot rows are contiguous in the workspace, so they arrive in shared memory
// by bulk copies of up to kMergeChunk slots. A chunk is then combined there:
// warp w takes slots w, w + 8, ..., lane l owns channels 4l .. 4l + 3.
// After the grid it depends on has finished, the merge costs one
// load round trip per chunk.
//
// The kernel triggers its dependents only after its wait: a later decode reuses the slots, and the
// chain append -> prologue -> decode lets that decode start only after this grid has finished.
//
// History slots hold attention over the stored (rotated) value basis. In
// explicit-V mode their combination is multiplied by R_V^T = P_br H U_V^T
// before it meets the BF16 slots, which are in the caller's basis (MarkTechPost
// article "Together AI 开源 OSCAR…", section "服务系统：混合精度缓存布局").
#include "kernels.cuh"
#include "rotate.cuh"
#include "tma.cuh"
#include "timeline.cuh"

namespace oscar {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;

// Fold slots [lo, hi) of the staged chunk (first slot c0) that belong to warp w
// (s = w mod kMergeWarps) into the warp's running (M, L, A); lane l owns
// channels 4l .. 4l + 3.
__device__ __forceinline__ void combine_part(const float* sbuf, int c0, int lo, int hi, int w, int lane, float& M,
                                             float& L, float4& A) {
  if (lo >= hi) return;
  const int first = lo + ((w - lo) % kMergeWarps + kMergeWarps) % kMergeWarps;
  float mx = -INFINITY;
  for (int s = first; s < hi; s += kMergeWarps) mx = fmaxf(mx, sbuf[(s - c0) * kPartFloats]);
  if (mx == -INFINITY) return;
  const float Mn = fmaxf(M, mx);
  const float r = (M == -INFINITY) ? 0.f : exp2f(M - Mn);
  L *= r;
  A.x *= r; A.y *= r; A.z *= r; A.w *= r;
  for (int s = first; s < hi; s += kMergeWarps) {
    const float* row = sbuf + (s - c0) * kPartFloats;
    const float m = row[0];
    if (m == -INFINITY) continue;
    const float wgt = exp2f(m - Mn);
    const float4 a = reinterpret_cast<const float4*>(row + 4)[lane];
    L = fmaf(row[1], wgt, L);
    A.x = fmaf(a.x, wgt, A.x);
    A.y = fmaf(a.y, wgt, A.y);
    A.z = fmaf(a.z, wgt, A.z);
    A.w = fmaf(a.w, wgt, A.w);
  }
  M = Mn;
}

// Combine the warps' (M, L, A[c]) of one part; M (the maximum over all warps) is
// the same in every thread, -inf when the part has no live slot.
__device__ __forceinline__ void combine_warps(const float* sm, const float* sl, const float (*sa)[kD], int c,
                                              float& M, float& L, float& A) {
  M = -INFINITY;
  L = A = 0.f;
#pragma unroll
  for (int i = 0; i < kMergeWarps; ++i) M = fmaxf(M, sm[i]);
  if (M == -INFINITY) return;
#pragma unroll
  for (int i = 0; i < kMergeWarps; ++i) {
    if (sm[i] == -INFINITY) continue;
    const float f = exp2f(sm[i] - M);
    L = fmaf(sl[i], f, L);
    if (c < kD) A = fmaf(sa[i][c], f, A);
  }
}

__global__ void __launch_bounds__(kMergeThreads, 1) k_merge(LayerView lv, DecodeWorkspace ws, int nsplit, int nbfs,
                                                         void* out, int out_dtype, float* lse) {
  TimelineSpan timeline_span(lv, kTlMerge);
  extern __shared__ __align__(128) float sbuf[];            // [kMergeChunk][kPartFloats]
  __shared__ __align__(8) uint64_t bar_mem;
  __shared__ float sm[2][kMergeWarps], sl[2][kMergeWarps];
  __shared__ __align__(16) float sa[2][kMergeWarps][kD];
  __shared__ float zbuf[kD];
  __shared__ int landed;
  const int hq = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const uint32_t bar = smem_addr(&bar_mem);
  if (tid == 0) {
    mbar_init(bar);
    landed = 1;
  }
  __syncthreads();
  pdl_wait();                                       // the partials are written by the preceding grid
  timeline_span.mark();
  // The decode grid is complete: the next kernel (typically the next layer's append, which itself waits
  // for this grid before it starts work) may be scheduled now.
  pdl_launch_dependents();
  const float* row0 = ws.partials + ((size_t)b * lv.hq + hq) * ws.nslots * kPartFloats;
  const int nslot = nsplit + nbfs;

  // per warp and part (history h, BF16 f): running (M, L, A) with L, A relative to 2^M
  float Mh = -INFINITY, Lh = 0.f, Mf = -INFINITY, Lf = 0.f;
  float4 Ah = make_float4(0.f, 0.f, 0.f, 0.f), Af = make_float4(0.f, 0.f, 0.f, 0.f);
  uint32_t phase = 0;
  for (int c0 = 0; c0 < nslot; c0 += kMergeChunk) {
    const int n = min(kMergeChunk, nslot - c0);
    if (tid == 0) bulk_load(smem_addr(sbuf), row0 + (size_t)c0 * kPartFloats, n * kPartFloats * 4, bar);
    if (!__syncthreads_and(mbar_wait(bar, phase))) {
      if (tid == 0) {
        flag(lv.status, OSCAR_STATUS_TIMEOUT);
        landed = 0;
      }
      mbar_wait(bar, phase);                        // one more bounded wait for the copy in flight
      break;
    }
    phase ^= 1u;
    combine_part(sbuf, c0, c0, min(c0 + n, nsplit), w, lane, Mh, Lh, Ah);       // history slots
    combine_part(sbuf, c0, max(c0, nsplit), c0 + n, w, lane, Mf, Lf, Af);       // BF16 slots
    __syncthreads();                                // chunk consumed before the buffer is refilled
  }
  if (lane == 0) {
    sm[0][w] = Mh; sl[0][w] = Lh;
    sm[1][w] = Mf; sl[1][w] = Lf;
  }
  *reinterpret_cast<float4*>(&sa[0][w][4 * lane]) = Ah;
  *reinterpret_cast<float4*>(&sa[1][w][4 * lane]) = Af;
  __syncthreads();

  // threads 0..127: channel c of both parts, the warps' states combined
  const int c = tid;
  float Mp0, Lp0, Ap0, Mp1, Lp1, Ap1;
  combine_warps(sm[0], sl[0], sa[0], c, Mp0, Lp0, Ap0);
  combine_warps(sm[1], sl[1], sa[1], c, Mp1, Lp1, Ap1);
  if (lv.v_explicit && Mp0 != -INFINITY && landed) {          // block-uniform condition
    // history part: rotated basis -> caller's basis, (a P_br H) U_V^T
    if (c < kD) zbuf[c] = Ap0;
    __syncthreads();
    float v[4];
    if (w == 0) {
#pragma unroll
      for (int r = 0; r < 4; ++r) v[r] = zbuf[rot_channel(lane, r)];   // (a P_br)[lane + 32 r]
      fwht128(v);
    }
    __syncthreads();
    if (w == 0) {
#pragma unroll
      for (int r = 0; r < 4; ++r) zbuf[lane + 32 * r] = v[r];
    }
    __syncthreads();
    if (c < kD) {
      const float* uvt = lv.params + (size_t)(hq / (lv.hq / lv.hkv)) * kParamFloats + kUVtOff;
      float o = 0.f;
#pragma unroll 8
      for (int i = 0; i < kD; ++i) o = fmaf(zbuf[i], __ldg(uvt + i * kD + c), o);   // (z U_V^T)[c]
      Ap0 = o;
    }
  }
  if (c >= kD) return;
  const float Mx = fmaxf(Mp0, Mp1);
  const float w0 = (Mp0 == -INFINITY) ? 0.f : exp2f(Mp0 - Mx);
  const float w1 = (Mp1 == -INFINITY) ? 0.f : exp2f(Mp1 - Mx);
  const float Ls = Lp0 * w0 + Lp1 * w1;
  const float o = (Ap0 * w0 + Ap1 * w1) * (1.f / Ls);
  const size_t oi = ((size_t)b * lv.hq + hq) * kD + c;
  if (out_dtype == OSCAR_OUT_FP32) static_cast<float*>(out)[oi] = o;
  else static_cast<__nv_bfloat16*>(out)[oi] = __float2bfloat16_rn(o);
  if (lse != nullptr && c == 0) lse[(size_t)b * lv.hq + hq] = (Mx + log2f(Ls)) * 0.6931471805599453f;
}

}  // namespace

int launch_merge(const LayerView& lv, const DecodeWorkspace& ws, int B, int nsplit, int nbfs, void* out,
                 int out_dtype, float* lse, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(lv.hq, B);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = kMergeChunk * kPartFloats * sizeof(float);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, k_merge, lv, ws, nsplit, nbfs, out, out_dtype, lse) != cudaSuccess)
    return OSCAR_ERR_CUDA;
  return OSCAR_OK;
}

int configure_merge_kernel() {
  return cudaFuncSetAttribute(k_merge, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kMergeChunk * kPartFloats * (int)sizeof(float)) == cudaSuccess
             ? OSCAR_OK
             : OSCAR_ERR_CUDA;
}

}  // namespace oscar
