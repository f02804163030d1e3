// Log-sum-exp merge of a decode call's partial results (sm_103a), shared by
// both decode algorithms (the news article "超越 TurboQuant…", section "OSCAR 的设计思路":
// the split partials are combined by an online softmax; partial = (m, l, acc) with l and acc
// relative to 2^m, m in log2 units).
//
// grid = (Hq, B), block = 256: one CTA per (request, query head). The head's
// slot rows are contiguous in the workspace, so they arrive in shared memory
// by bulk copies of up to kMergeChunk slots. A chunk is then combined by block
// reductions: the maxima per part, one weight per slot (one thread each), the
// l sums, and per output channel one pass over the slots (two threads per
// channel, one half of the slots each). After the grid it depends on has
// finished, the merge costs one load round trip per chunk.
//
// The kernel triggers its dependents only after its wait: a later decode reuses the slots, and the
// chain append -> prologue -> decode lets that decode start only after this grid has finished.
//
// History slots hold attention over the stored (rotated) value basis. In
// explicit-V mode their combination is multiplied by R_V^T = P_br H U_V^T
// before it meets the BF16 slots, which are in the caller's basis (MarkTechPost
// article "Together AI 开源 OSCAR…", section "服务系统：混合精度缓存布局").
#include <algorithm>

#include "kernels.cuh"
#include "rotate.cuh"
#include "tma.cuh"
#include "timeline.cuh"

namespace oscar {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;

// 2^x with the SFU (x <= 0 or -inf here)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Block-wide max (op 0) or sum (op 1) of two values over NW warps; every thread gets the results.
template <int OP, int NW = kMergeWarps>
__device__ __forceinline__ float2 block_reduce2(float2 v, float2* red) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int x = 16; x > 0; x >>= 1) {
    const float a = __shfl_xor_sync(0xffffffffu, v.x, x), b = __shfl_xor_sync(0xffffffffu, v.y, x);
    v.x = OP == 0 ? fmaxf(v.x, a) : v.x + a;
    v.y = OP == 0 ? fmaxf(v.y, b) : v.y + b;
  }
  __syncthreads();                                  // red[] free from its previous use
  if (lane == 0) red[w] = v;
  __syncthreads();
  float2 r = red[0];
#pragma unroll
  for (int i = 1; i < NW; ++i) {
    r.x = OP == 0 ? fmaxf(r.x, red[i].x) : r.x + red[i].x;
    r.y = OP == 0 ? fmaxf(r.y, red[i].y) : r.y + red[i].y;
  }
  return r;
}

__global__ void __launch_bounds__(kMergeThreads, 1) k_merge(LayerView lv, DecodeWorkspace ws, int nsplit, int nbfs,
                                                            void* out, int out_dtype, float* lse) {
  TimelineSpan timeline_span(lv, kTlMerge);
  extern __shared__ __align__(128) float sbuf[];            // [min(kMergeChunk, slots)][kPartFloats]
  __shared__ __align__(8) uint64_t bar_mem;
  __shared__ float2 red[kMergeWarps];
  __shared__ float wts[kMergeChunk];
  __shared__ float ahalf[2][kD];
  __shared__ float zbuf[kD];
  __shared__ int landed;
  const int hq = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int c = tid & (kD - 1), half = tid >> 7;            // output channel, slot half of this thread
  const uint32_t bar = smem_addr(&bar_mem);
  if (tid == 0) {
    mbar_init(bar);
    landed = 1;
  }
  __syncthreads();
  pdl_wait();                                       // the partials are written by the preceding grid
  timeline_span.mark();
  // The decode grid is complete: the next kernel (typically the next layer's prologue, which itself waits
  // for this grid before it starts work) may be scheduled now.
  pdl_launch_dependents();
  const float* row0 = ws.partials + ((size_t)b * lv.hq + hq) * ws.nslots * kPartFloats;
  const int nslot = nsplit + nbfs;

  // running state per part (x: history slots, y: BF16 slots): M and L are block-uniform, A is this
  // thread's channel c summed over its half of the slots; L and A are relative to 2^M
  float2 M = make_float2(-INFINITY, -INFINITY), L = make_float2(0.f, 0.f), A = make_float2(0.f, 0.f);
  uint32_t phase = 0;
  const int chunk = min(kMergeChunk, nslot);       // slots per bulk copy; the launch sized sbuf for it
  for (int c0 = 0; c0 < nslot; c0 += chunk) {
    const int n = min(chunk, nslot - c0);
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
    // 1. the chunk's maxima per part; rescale the running state
    const bool mine = tid < n;
    const bool hist = c0 + tid < nsplit;
    const float m = mine ? sbuf[tid * kPartFloats] : -INFINITY;
    const float2 cm = block_reduce2<0>(make_float2(hist ? m : -INFINITY, hist ? -INFINITY : m), red);
    const float2 Mn = make_float2(fmaxf(M.x, cm.x), fmaxf(M.y, cm.y));
    const float2 r = make_float2(M.x == -INFINITY ? 0.f : ex2(M.x - Mn.x), M.y == -INFINITY ? 0.f : ex2(M.y - Mn.y));
    L = make_float2(L.x * r.x, L.y * r.y);
    A = make_float2(A.x * r.x, A.y * r.y);
    M = Mn;
    // 2. one weight per slot, and the chunk's l sums
    float wt = 0.f;
    if (mine && m != -INFINITY) wt = ex2(m - (hist ? M.x : M.y));
    if (tid < kMergeChunk) wts[tid] = wt;
    const float lw = mine ? sbuf[tid * kPartFloats + 1] * wt : 0.f;
    const float2 cl = block_reduce2<1>(make_float2(hist ? lw : 0.f, hist ? 0.f : lw), red);   // also publishes wts
    L = make_float2(L.x + cl.x, L.y + cl.y);
    // 3. channel c over this thread's half of the chunk: history slots [0, nh), BF16 slots [nh, n)
    const int nh = max(0, min(n, nsplit - c0));
    const int mid = (n + 1) >> 1, s_lo = half ? mid : 0, s_hi = half ? n : mid;
    float ax = 0.f, ay = 0.f;
#pragma unroll 4
    for (int t = s_lo; t < min(s_hi, nh); ++t) ax = fmaf(wts[t], sbuf[t * kPartFloats + 4 + c], ax);
#pragma unroll 4
    for (int t = max(s_lo, nh); t < s_hi; ++t) ay = fmaf(wts[t], sbuf[t * kPartFloats + 4 + c], ay);
    A = make_float2(A.x + ax, A.y + ay);
    __syncthreads();                                // the chunk is consumed before the buffer is refilled
  }
  // the two halves of every channel
  if (half == 1) {
    ahalf[0][c] = A.x;
    ahalf[1][c] = A.y;
  }
  __syncthreads();
  float Ah = A.x + ahalf[0][c], Af = A.y + ahalf[1][c];
  if (lv.v_explicit && M.x != -INFINITY && landed) {          // block-uniform condition
    // history part: rotated basis -> caller's basis, (a P_br H) U_V^T
    if (half == 0) zbuf[c] = Ah;
    __syncthreads();
    float v[4];
    if (w == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = zbuf[rot_channel(lane, q)];   // (a P_br)[lane + 32 q]
      fwht128(v);
    }
    __syncthreads();
    if (w == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) zbuf[lane + 32 * q] = v[q];
    }
    __syncthreads();
    if (half == 0) {
      const float* uvt = lv.params + (size_t)(hq / (lv.hq / lv.hkv)) * kParamFloats + kUVtOff;
      float o = 0.f;
#pragma unroll 8
      for (int i = 0; i < kD; ++i) o = fmaf(zbuf[i], __ldg(uvt + i * kD + c), o);   // (z U_V^T)[c]
      Ah = o;
    }
  }
  if (half == 1) return;
  const float Mx = fmaxf(M.x, M.y);
  const float w0 = (M.x == -INFINITY) ? 0.f : exp2f(M.x - Mx);
  const float w1 = (M.y == -INFINITY) ? 0.f : exp2f(M.y - Mx);
  const float Ls = L.x * w0 + L.y * w1;
  const float o = (Ah * w0 + Af * w1) * (1.f / Ls);
  const size_t oi = ((size_t)b * lv.hq + hq) * kD + c;
  if (out_dtype == OSCAR_OUT_FP32) static_cast<float*>(out)[oi] = o;
  else static_cast<__nv_bfloat16*>(out)[oi] = __float2bfloat16_rn(o);
  if (lse != nullptr && c == 0) lse[(size_t)b * lv.hq + hq] = (Mx + log2f(Ls)) * 0.6931471805599453f;
}


// V-absorbed mode: no rotation follows the combination, so the channels split
// across kMergeParts CTAs per (request, query head) of 128 threads. Lane l of
// warp w owns channel 32 part + l and the slots w, w + 4, ... of a chunk of
// kMergeSplitChunk slots; each slot row's 32 channels are one coalesced 128-byte
// load, and a chunk's loads (headers and values) are all issued before the first
// reduction, so a chunk costs one load round trip. 128 threads keep the CTA
// small enough to be scheduled beside the decode CTAs it waits for.
constexpr int kMergeParts = 4;
constexpr int kMergeSplitThreads = 128;
constexpr int kMergeSplitWarps = kMergeSplitThreads / 32;
constexpr int kMergeSplitChunk = 64;
constexpr int kMergeSplitPer = kMergeSplitChunk / kMergeSplitWarps;   // slots per thread and chunk

__global__ void __launch_bounds__(kMergeSplitThreads) k_merge_split(LayerView lv, DecodeWorkspace ws, int nsplit,
                                                                    int nbfs, void* out, int out_dtype, float* lse) {
  TimelineSpan timeline_span(lv, kTlMerge);
  __shared__ float2 red[kMergeSplitWarps];
  __shared__ float wts[kMergeSplitChunk];
  __shared__ float2 accs[kMergeSplitWarps][32];
  const int hq = blockIdx.x, b = blockIdx.y, part = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int c = 32 * part + lane;                   // output channel of this thread
  pdl_wait();                                       // the partials are written by the preceding grid
  timeline_span.mark();
  pdl_launch_dependents();                          // as in k_merge: only after the wait
  const float* row0 = ws.partials + ((size_t)b * lv.hq + hq) * ws.nslots * kPartFloats;
  const int nslot = nsplit + nbfs;
  // running state per part (x: history slots, y: BF16 slots), relative to 2^M
  float2 M = make_float2(-INFINITY, -INFINITY), L = make_float2(0.f, 0.f), A = make_float2(0.f, 0.f);
  for (int c0 = 0; c0 < nslot; c0 += kMergeSplitChunk) {
    const int n = min(kMergeSplitChunk, nslot - c0);
    float m = -INFINITY, l = 0.f;
    if (tid < n) {
      const float2 ml = *reinterpret_cast<const float2*>(row0 + (size_t)(c0 + tid) * kPartFloats);
      m = ml.x;
      l = ml.y;
    }
    float v[kMergeSplitPer];
#pragma unroll
    for (int i = 0; i < kMergeSplitPer; ++i) {
      const int sl = w + kMergeSplitWarps * i;
      v[i] = sl < n ? row0[(size_t)(c0 + sl) * kPartFloats + 4 + c] : 0.f;
    }
    // the chunk's maxima per part; rescale the running state
    const bool hist = c0 + tid < nsplit;
    const float2 cm = block_reduce2<0, kMergeSplitWarps>(make_float2(hist ? m : -INFINITY, hist ? -INFINITY : m), red);
    const float2 Mn = make_float2(fmaxf(M.x, cm.x), fmaxf(M.y, cm.y));
    const float2 r = make_float2(M.x == -INFINITY ? 0.f : ex2(M.x - Mn.x), M.y == -INFINITY ? 0.f : ex2(M.y - Mn.y));
    L = make_float2(L.x * r.x, L.y * r.y);
    A = make_float2(A.x * r.x, A.y * r.y);
    M = Mn;
    // one weight per slot (thread tid < n), and the chunk's l sums
    float wt = 0.f;
    if (tid < n && m != -INFINITY) wt = ex2(m - (hist ? M.x : M.y));
    if (tid < kMergeSplitChunk) wts[tid] = wt;
    const float lw = tid < n ? l * wt : 0.f;
    const float2 cl = block_reduce2<1, kMergeSplitWarps>(make_float2(hist ? lw : 0.f, hist ? 0.f : lw), red);
    L = make_float2(L.x + cl.x, L.y + cl.y);        // the reduction's barriers also published wts
#pragma unroll
    for (int i = 0; i < kMergeSplitPer; ++i) {
      const int sl = w + kMergeSplitWarps * i;
      if (sl < n) {
        if (c0 + sl < nsplit) A.x = fmaf(wts[sl], v[i], A.x);
        else A.y = fmaf(wts[sl], v[i], A.y);
      }
    }
    __syncthreads();                                // wts is rewritten by the next chunk
  }
  accs[w][lane] = A;
  __syncthreads();
  if (w != 0) return;
  float Ah = 0.f, Af = 0.f;
#pragma unroll
  for (int ww = 0; ww < kMergeSplitWarps; ++ww) {
    Ah += accs[ww][lane].x;
    Af += accs[ww][lane].y;
  }
  const float Mx = fmaxf(M.x, M.y);
  const float w0 = (M.x == -INFINITY) ? 0.f : exp2f(M.x - Mx);
  const float w1 = (M.y == -INFINITY) ? 0.f : exp2f(M.y - Mx);
  const float Ls = L.x * w0 + L.y * w1;
  const float o = (Ah * w0 + Af * w1) * (1.f / Ls);
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
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (!lv.v_explicit) {                             // channels split across CTAs
    cfg.gridDim = dim3(lv.hq, B, kMergeParts);
    cfg.blockDim = dim3(kMergeSplitThreads);
    cfg.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&cfg, k_merge_split, lv, ws, nsplit, nbfs, out, out_dtype, lse);
  } else {                                          // whole rows: the rotation back needs every channel
    cfg.gridDim = dim3(lv.hq, B);
    cfg.blockDim = dim3(kMergeThreads);
    // only the slots one copy brings: a smaller footprint lets the grid sit beside the decode CTAs it waits for
    cfg.dynamicSmemBytes = std::min(kMergeChunk, nsplit + nbfs) * kPartFloats * sizeof(float);
    e = cudaLaunchKernelEx(&cfg, k_merge, lv, ws, nsplit, nbfs, out, out_dtype, lse);
  }
  return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int configure_merge_kernel() {
  if (cudaFuncSetAttribute(k_merge, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kMergeChunk * kPartFloats * (int)sizeof(float)) != cudaSuccess)
    return OSCAR_ERR_CUDA;
  if (set_max_shared_carveout(reinterpret_cast<const void*>(k_merge)) != OSCAR_OK) return OSCAR_ERR_CUDA;
  return set_max_shared_carveout(reinterpret_cast<const void*>(k_merge_split));
}

}  // namespace oscar
