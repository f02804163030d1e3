// Query prologue of the decode (sm_103a): q~ = q R_K for the query heads of
// one (request, kv head) group, and everything the history kernels read
// about it (MarkTechPost article "Together AI 开源 OSCAR…", section "OSCAR 有何
// 不同做法": R_K = U_Q H_Had P_br; the read path's inverse rotation of the
// keys is applied once to the query instead, R_K being orthogonal).
//
// Outputs, per query head:
//  * ws.qrot  : q~ in rotated channel order (float32), for the CUDA-core kernel;
//  * ws.qconst: group sums of q~, F = sm_scale log2(e) 2^-sigma, the scaled group
//               sums (zero-point terms), the fragment offsets and sigma;
//  * ws.qfrag : fp16 B fragments of the tensor-core logits. The tensor-core
//               kernel feeds code c of channel ch as the fp16 subnormal
//               c W(ch) 2^-24, W(ch) = 4^(p mod 4) for the code's position p in
//               its 16-bit half of the packed word (the masked bits themselves,
//               after a shift by 8 for p >= 4). With x(ch) = q~[ch] 2^sigma / W(ch)
//               split into two fp16 parts hi = fp16(x), lo = fp16(x - hi), the
//               fragments carry hi and lo in separate columns; summing both,
//               sum_{ch in g} c W(ch) 2^-24 (hi + lo)(ch) = 2^(sigma - 24) sum c q~
//               to about 22 bits, with no constant part to cancel (the offsets
//               below are 0). Codebook pools feed the level k_c the same way, as
//               the fp16 subnormal k_c 2^-24.
//               k-block kb = 4 G + j (G the channel group) at lane (g', t') holds
//               k rows (2t', 2t'+1) -> channels (c0, c0 + 8) and (2t'+8, 2t'+9) ->
//               channels (c0 + 1, c0 + 9), c0 = 16 (t' + 4 G) + 2 j; column g' is
//               (head 4 nt + g'/2, part g'%2). sigma puts max|q~| near 2^12.
//               Codebook pools (OSCAR_META_CB): the kernel feeds level k_c as k_c 2^-24
//               (W = 1 for every channel), k rows (2t', 2t'+1) -> channels (c0, c0 + 4) and
//               (2t'+8, 2t'+9) -> channels (c0 + 8, c0 + 12), c0 = 16 (t' + 4 G) + j.
#pragma once

#include "kernels.cuh"
#include "rotate.cuh"
#include "tma.cuh"

namespace oscar {

// fp16 rounding of a fragment value, subnormal results flushed to zero so that
// nothing depends on how the tensor cores treat fp16 subnormal inputs.
__device__ __forceinline__ float frag_round(float x) {
  const float r = __half2float(__float2half_rn(x));
  return fabsf(r) < 6.103515625e-05f ? 0.f : r;
}

// One 16-row tile of fp32 rows (smem, [16][kTileStride], rows[i * kTileStride + c]) times the
// composite rotation R = U H P_br on the tensor cores. R arrives in shared
// memory as fp16 high + low parts in mma.m16n8k16 B-fragment order (frag_s,
// 64 KB, its 8 k-block chunks of 8 KB completing on mbarriers bars + 8 kb).
// A = the rows as fp16; one fresh accumulator per k-block, added in rounding
// fp32 (the tensor cores' accumulation truncates). Warp w of 8 takes n-tiles 2w
// and 2w + 1, i.e. rotated channels 16 w .. 16 w + 15. On return (after a block
// barrier) every row of `rows` holds its rotation in rotated channel order.
// Returns false (block-uniform) when a chunk never landed; rows are then
// unchanged.
constexpr int kPrologueWarps = 8;
__device__ __forceinline__ void qp_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                       uint32_t b0, uint32_t b1, bool zero_c) {
  if (zero_c)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Row stride of the fp32 tiles: 136 floats makes the 64-bit fragment loads of
// rows g = 0..7 (stride 68 eight-byte words, 68 = 4 mod 16) conflict-free.
constexpr int kTileStride = kD + 8;

__device__ __forceinline__ uint32_t f16x2_of(const float* x) {
  const float2 p = *reinterpret_cast<const float2*>(x);
  const __half2 v = __floats2half2_rn(p.x, p.y);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ bool rotate_tile16(const uint32_t* frag_s, float* rows, uint32_t bars) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  uint32_t a[8][4];
#pragma unroll
  for (int kb = 0; kb < 8; ++kb) {
    const float* r0 = rows + g * kTileStride + 16 * kb + 2 * t;
    const float* r8 = rows + (g + 8) * kTileStride + 16 * kb + 2 * t;
    a[kb][0] = f16x2_of(r0);           // row g, channels 16 kb + 2t, +1
    a[kb][1] = f16x2_of(r8);           // row g + 8
    a[kb][2] = f16x2_of(r0 + 8);       // row g, channels 16 kb + 2t + 8, +9
    a[kb][3] = f16x2_of(r8 + 8);
  }
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  bool landed = true;
#pragma unroll
  for (int kb = 0; kb < 8; ++kb) {
    landed = landed && mbar_wait(bars + 8 * kb, 0);
    if (!landed) break;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint4 f = *reinterpret_cast<const uint4*>(frag_s + ((kb * 16 + 2 * w + j) * 32 + lane) * 4);
      float d[4];
      qp_mma(d, a[kb][0], a[kb][1], a[kb][2], a[kb][3], f.x, f.y, true);    // x R_hi
      qp_mma(d, a[kb][0], a[kb][1], a[kb][2], a[kb][3], f.z, f.w, false);   // + x R_lo
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] += d[e];
    }
  }
  if (!__syncthreads_and(landed)) return false;        // also: every warp has read its A rows
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int col = 8 * (2 * w + j) + 2 * t;            // rotated channel
    *reinterpret_cast<float2*>(rows + g * kTileStride + col) = make_float2(acc[j][0], acc[j][1]);
    *reinterpret_cast<float2*>(rows + (g + 8) * kTileStride + col) = make_float2(acc[j][2], acc[j][3]);
  }
  __syncthreads();
  return true;
}

// Per query head qi of group (b, h) (warp w takes heads w, w + nwarps, ...):
// q~ (xs[qi * stride + 0..127], rotated channel order) goes to the workspace with its
// group sums, and sig[qi] = sigma, the power of two that brings max|q~| near 2^12.
__device__ __forceinline__ void qprep_stats(const LayerView& lv, const DecodeWorkspace& ws, const float* xs,
                                            int stride, int* sig, int b, int h, int nwarps) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lv.hq / lv.hkv;
  for (int qi = w; qi < gq; qi += nwarps) {
    const int hq = h * gq + qi;
    float* dst = ws.qrot + ((size_t)b * lv.hq + hq) * kD;
    float y[4], mx = 0.f;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      y[r] = xs[qi * stride + lane + 32 * r];
      dst[lane + 32 * r] = y[r];
      mx = fmaxf(mx, fabsf(y[r]));
    }
    float s0 = y[0] + y[1], s1 = y[2] + y[3];           // channels 0..63: group 0
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, m);
      s1 += __shfl_xor_sync(0xffffffffu, s1, m);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    }
    if (lane == 0) {
      float* qc = ws.qconst + ((size_t)b * lv.hq + hq) * kQConst;
      qc[kQSum0] = s0;
      qc[kQSum1] = s1;
      int e = 0;
      if (mx > 0.f && isfinite(mx)) frexpf(mx, &e);  // mx in [2^(e-1), 2^e)
      sig[qi] = min(max(12 - e, -60), 60);
    }
  }
}

// 2^e for |e| < 126, built from its bits
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }

// After qprep_stats and a barrier of the participating warps 0 .. nwarps-1:
// per-head constants (warp w handles heads w, w + nwarps, ...; lane l owns
// channels 4l .. 4l + 3) and the fragments (all participating threads). q~ of
// head qi is xs[qi * stride + 0..127].
__device__ __forceinline__ void qprep_finish(const LayerView& lv, const DecodeWorkspace& ws, const float* xs,
                                             int stride, const int* sig, int b, int h, float scale_log2,
                                             int nwarps) {
  const int tid = threadIdx.x, wib = tid >> 5, lane = tid & 31;
  const int gq = lv.hq / lv.hkv;
  for (int qi = wib; qi < gq; qi += nwarps) {
    const float sc = pow2i(sig[qi]);
    float offh = 0.f, offl = 0.f, sum = 0.f;       // the offsets stay 0: no operand carries a constant part
    (void)sc;
#pragma unroll
    for (int e = 0; e < 4; ++e) sum += xs[qi * stride + 4 * lane + e];   // channel 4 lane + e
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) {              // lanes 0..15 hold group 0, 16..31 group 1
      offh += __shfl_xor_sync(0xffffffffu, offh, m);
      offl += __shfl_xor_sync(0xffffffffu, offl, m);
      sum += __shfl_xor_sync(0xffffffffu, sum, m);
    }
    float* qc = ws.qconst + ((size_t)b * lv.hq + h * gq + qi) * kQConst;
    if (lane == 0 || lane == 16) {
      const int g = lane >> 4;
      qc[g ? kQZ1 : kQZ0] = scale_log2 * sum;
      qc[g ? kQOff1H : kQOff0H] = 1024.f * offh;
      qc[g ? kQOff1L : kQOff0L] = 1024.f * offl;
    }
    if (lane == 0) {
      qc[kQF] = scale_log2 * pow2i(-sig[qi]);
      qc[kQSigma] = (float)sig[qi];
    }
  }
  const int nt_count = (gq + 3) / 4;
  uint32_t* frag = ws.qfrag + ((size_t)b * lv.hkv + h) * kFragWords;
  for (int wi = tid; wi < 8 * 2 * 64; wi += nwarps * 32) {
    const int r = wi & 1, lp = (wi >> 1) & 31, nt = (wi >> 6) & 1, kb = wi >> 7;
    const int gp = lp >> 2, tp = lp & 3;
    const int head = 4 * nt + (gp >> 1), part = gp & 1;
    uint32_t word = 0;
    if (nt < nt_count && head < gq) {
      // r = 0: channels (c0, c0 + 8), code position p = 2 (kb & 3) in its 16-bit half; r = 1: (c0 + 1,
      // c0 + 9), p + 1. The code of position p is fed as c 4^(p mod 4) 2^-24, so the fragment carries
      // q~ 2^sigma / 4^(p mod 4) (the kernel's F takes the 2^24). Codebook pools: r = 0: (c0, c0 + 4),
      // r = 1: (c0 + 8, c0 + 12), levels fed as k_c 2^-24 (W = 1).
      const float sc = lv.meta_cb ? pow2i(sig[head]) : pow2i(sig[head] - 2 * ((2 * (kb & 3) + r) & 3));
      const int c0 = lv.meta_cb ? 16 * (tp + 4 * (kb >> 2)) + (kb & 3) + 8 * r
                                : 16 * (tp + 4 * (kb >> 2)) + 2 * (kb & 3) + r;
      const int c1 = c0 + (lv.meta_cb ? 4 : 8);
      float x[2] = {xs[head * stride + c0] * sc, xs[head * stride + c1] * sc};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float hi = frag_round(x[e]);
        x[e] = part ? frag_round(x[e] - hi) : hi;
      }
      const __half2 v = __floats2half2_rn(x[0], x[1]);
      word = *reinterpret_cast<const uint32_t*>(&v);
    }
    frag[((kb * 2 + nt) * 32 + lp) * 2 + r] = word;
  }
}

}  // namespace oscar
