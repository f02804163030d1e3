// Warp-level rotation x -> x U H_Had P_br and the INT2 quantiser (sm_103a).
//
// Rotation (MarkTechPost article "Together AI 开源 OSCAR…", section "OSCAR 有何不同
// 做法": R = U H_Had P_br). One warp handles one 128-channel row: the dense
// product with U, then a warp-shuffle fast Walsh-Hadamard transform, then the
// bit-reversal permutation, which is never materialised: lane l, slot r holds
// pre-permutation element i = l + 32 r, and that element lands in rotated
// channel bitrev7(i). For d = 128 this gives
//     rotated channel  j = (rev5(l) << 2) | rev2(r)
//     group            j >> 6 = l & 1
//     packed byte      j >> 2 = rev5(l)     (each lane owns one byte of the row)
//     bit position     2 * (j & 3) = 2 * rev2(r)
//
// Quantiser (same article, "服务系统：混合精度缓存布局": clip to per-channel
// thresholds, per-token asymmetric INT2 over 64-channel groups). The steps are
// single IEEE float32 operations in a fixed order so the codes are exactly
// reproducible: clip, group min/max, scale = (max - min) / 3, fp16 (RNE,
// saturating) scale and zero = min, code = rint((y - zero') / scale') clamped
// to [0, 3] using the stored fp16 scale' and zero'; scale' == 0 gives code 0.
#pragma once

#include "common.cuh"

namespace oscar {

__device__ __forceinline__ int rev5(int l) { return (int)(__brev((unsigned)l) >> 27); }
__device__ __forceinline__ int rev2(int r) { return ((r & 1) << 1) | (r >> 1); }
__device__ __forceinline__ int rot_channel(int lane, int r) { return (rev5(lane) << 2) | rev2(r); }

// In-warp Walsh-Hadamard transform of 128 values, lane holds v[r] = element lane + 32 r.
// Output is orthonormal (scaled by 1/sqrt(128)), still in pre-permutation order.
__device__ __forceinline__ void fwht128(float (&v)[4]) {
  const int lane = threadIdx.x & 31;
  float a0 = v[0] + v[1], a1 = v[0] - v[1];     // stride 32 (r bit 0)
  float a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2; v[2] = a0 - a2;               // stride 64 (r bit 1)
  v[1] = a1 + a3; v[3] = a1 - a3;
#pragma unroll
  for (int s = 1; s < 32; s <<= 1) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float o = __shfl_xor_sync(0xffffffffu, v[r], s);
      v[r] = (lane & s) ? (o - v[r]) : (v[r] + o);
    }
  }
  const float inv = 0.08838834764831845f;       // 1/sqrt(128)
#pragma unroll
  for (int r = 0; r < 4; ++r) v[r] *= inv;
}

// Rotate T rows. xs: T rows of 128 floats (shared memory, read as broadcasts);
// U: row-major [128][128] float (shared or global). On return y[t][r] is the
// rotated value of channel rot_channel(lane, r) of row t.
template <int T>
__device__ __forceinline__ void warp_rotate(const float* __restrict__ U, const float* xs, float (&y)[T][4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < T; ++t)
#pragma unroll
    for (int r = 0; r < 4; ++r) y[t][r] = 0.f;
#pragma unroll 4
  for (int i = 0; i < kD; ++i) {
    const float* row = U + i * kD + lane;
    float u0 = row[0], u1 = row[32], u2 = row[64], u3 = row[96];
#pragma unroll
    for (int t = 0; t < T; ++t) {
      float xi = xs[t * kD + i];
      y[t][0] = fmaf(xi, u0, y[t][0]);
      y[t][1] = fmaf(xi, u1, y[t][1]);
      y[t][2] = fmaf(xi, u2, y[t][2]);
      y[t][3] = fmaf(xi, u3, y[t][3]);
    }
  }
#pragma unroll
  for (int t = 0; t < T; ++t) fwht128(y[t]);
}

__device__ __forceinline__ float sat_fp16(float x) { return fminf(fmaxf(x, -65504.f), 65504.f); }

// Quantise one rotated row held as y[r] (channel rot_channel(lane, r)) and
// write its packed byte and group metadata into the page block `blk`, row
// `row`, half `kind` (OSCAR_KIND_K / OSCAR_KIND_V). tau: float [128] clip
// thresholds indexed by rotated channel. mc: null for the fp16 (scale, zero) metadata, else the
// kind's compact-format constants {T, D, E, 0} for groups 0 and 1 (8 floats). cb: null, or the kind's
// codebook constants {k_0..k_3, theta_0..theta_2, 0} (codebook format: fp16 range and zero).
// status: when not null, OSCAR_STATUS_NONFINITE is flagged for a non-finite input value and
// OSCAR_STATUS_SATURATED for fp16 metadata stored saturated.
__device__ __forceinline__ void quantize_pack_row(const float (&y_in)[4], const float* __restrict__ tau,
                                                  uint8_t* blk, int row, int kind, const float* __restrict__ mc,
                                                  const float* __restrict__ cb = nullptr, int* status = nullptr) {
  const int lane = threadIdx.x & 31;
  bool bad = false;
#pragma unroll
  for (int r = 0; r < 4; ++r) bad |= nonfinite(y_in[r]);
  float y[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    float t = tau[rot_channel(lane, r)];
    y[r] = fminf(fmaxf(y_in[r], -t), t);
  }
  float mn = fminf(fminf(y[0], y[1]), fminf(y[2], y[3]));
  float mx = fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3]));
#pragma unroll
  for (int s = 2; s < 32; s <<= 1) {            // lanes of equal parity share a group
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, s));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
  }
  float sq, zq;
  __half s16, z16;
  unsigned mn8 = 0, mx8 = 0;
  if (mc == nullptr) {
    const float diff = __fsub_rn(mx, mn);
    const float scale = cb != nullptr ? diff : __fdiv_rn(diff, 3.0f);   // codebook format: the range
    if (status != nullptr && (fp16_saturates(scale) || fp16_saturates(mn)) && (lane & 30) == 0)
      flag(status, OSCAR_STATUS_SATURATED);
    s16 = __float2half_rn(sat_fp16(scale));
    z16 = __float2half_rn(sat_fp16(mn));
    sq = __half2float(s16);
    zq = __half2float(z16);
  } else {
    const float* c = mc + 4 * (lane & 1);           // lanes of group (lane & 1)
    u8_quant_params(mn, mx, c[0], c[1], c[2], mn8, mx8, sq, zq);
  }
  unsigned byte = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    float c = 0.f;
    if (sq != 0.f) {
      const float t = __fdiv_rn(__fsub_rn(y[r], zq), sq);
      c = cb != nullptr ? cb_code(t, cb) : fminf(fmaxf(rintf(t), 0.f), 3.f);
    }
    byte |= ((unsigned)c) << (2 * rev2(r));
  }
  if (status != nullptr && __any_sync(0xffffffffu, bad) && lane == 0) flag(status, OSCAR_STATUS_NONFINITE);
  const int b = rev5(lane);
  if (kind == OSCAR_KIND_K) {
    blk[kKCodesOff + row * (kD / 4) + b] = (uint8_t)byte;
  } else {                                       // channel-major: one 2-bit field per channel
#pragma unroll
    for (int r = 0; r < 4; ++r) v_set_code(blk, rot_channel(lane, r), row, (byte >> (2 * rev2(r))) & 3u);
  }
  if (lane < 2) {                                // lane 0: group 0, lane 1: group 1
    if (mc == nullptr) {
      __half2 sz = __halves2half2(s16, z16);
      const int off = (kind == OSCAR_KIND_K ? kKMetaOff : kVMetaOff) + row * (kNG * 4) + lane * 4;
      *reinterpret_cast<__half2*>(blk + off) = sz;
    } else {
      const int off = (kind == OSCAR_KIND_K ? kKMetaOff : kVMetaOffU8) + row * (kNG * 2) + lane * 2;
      *reinterpret_cast<uint16_t*>(blk + off) = (uint16_t)(mn8 | (mx8 << 8));
    }
  }
}

}  // namespace oscar
