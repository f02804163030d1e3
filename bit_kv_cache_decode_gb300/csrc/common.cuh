// Shared device definitions of the OSCAR INT2 KV-cache library (sm_103a).
//
// Geometry of the mixed-precision token pool (news article "超越 TurboQuant…
// Together AI 最新论文 OSCAR…", section "OSCAR 的设计思路": BF16 sink | INT2
// history | BF16 recent, 4 two-bit codes per byte; MarkTechPost article
// "Together AI 开源 OSCAR…", section "服务系统：混合精度缓存布局": 64-channel
// groups, per-token asymmetric INT2).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/oscar.h"

namespace oscar {

constexpr int kD = 128;                       // head_dim
constexpr int kG = 64;                        // channels per quantisation group
constexpr int kNG = kD / kG;                  // groups per token row
constexpr int kP = 64;                        // tokens per page
constexpr int kCodeBytes = kP * kD / 4;       // 2048: K (or V) codes of a page block
constexpr int kMetaBytes = kP * kNG * 4;      // 512: fp16 (scale, zero) per group per row
constexpr int kKCodesOff = 0;
constexpr int kVCodesOff = kCodeBytes;
constexpr int kKMetaOff = 2 * kCodeBytes;
constexpr int kVMetaOff = 2 * kCodeBytes + kMetaBytes;
constexpr int kBlockBytes = 2 * kCodeBytes + 2 * kMetaBytes;   // 5120
// Compact metadata (OSCAR_META_U8, 16 bits per group: the pages' 2.25 bits per history element):
// per row and group the bytes (mn8, mx8), indices on a grid of 255 steps over [-T, T], T the
// group's largest clip threshold. K metadata at kKMetaOff, V metadata right after it.
constexpr int kMetaBytesU8 = kP * kNG * 2;                       // 256
constexpr int kVMetaOffU8 = 2 * kCodeBytes + kMetaBytesU8;       // 4352
constexpr int kBlockBytesU8 = 2 * kCodeBytes + 2 * kMetaBytesU8; // 4608
// metadata formats as kernel template arguments (OSCAR_META_F16 / _U8 / _CB)
constexpr int kFmtF16 = 0, kFmtU8 = 1, kFmtCB = 2;
constexpr int kBf16BlockBytes = 2 * kP * kD * 2;               // 32768: K [P][D] then V [P][D]
// rotation parameters per kv head (float32 words): U_K [D][D], U_V [D][D], U_V transposed [D][D]
// (for coalesced reads of R_V^T in the merge), tau_K [D], tau_V [D], then the composite
// rotations R_K = U_K H P_br and R_V (explicit-V mode) as fp16 high + low parts in tensor-core
// B-fragment order for the prefill and the query prologue (kRFragWords 32-bit words each, see
// set_rotation)
constexpr int kRFragWords = 8 * 16 * 32 * 4;  // [k-block 8][n-tile 16][lane 32][hi b0, hi b1, lo b0, lo b1]
constexpr int kUKOff = 0, kUVOff = kD * kD, kUVtOff = 2 * kD * kD, kTauKOff = 3 * kD * kD,
              kTauVOff = 3 * kD * kD + kD, kRKFragOff = 3 * kD * kD + 2 * kD, kRVFragOff = kRKFragOff + kRFragWords;
// then, per kind and group, the compact format's grid constants {T, D = fl32(2T / 255), E = fl32(D / 3),
// 0}, and per kind the codebook {k_0, k_1, k_2, k_3, theta_0, theta_1, theta_2, 0} as floats
// (kMetaCFloats words, padded so that a head's parameters stay 128-byte aligned)
constexpr int kMetaCOff = kRVFragOff + kRFragWords, kCbOff = kMetaCOff + 16, kMetaCFloats = 32;
// then R_K and R_V (explicit-V mode) as three bf16 parts (R = b1 + b2 + b3, about 24 significant bits),
// each part the tensor-core B operand of the bulk prefill as it sits in shared memory: [part 3][k half 2]
// [n 128][128 bytes], K-major with the 128-byte swizzle (the 16-byte chunk j of row n at j ^ (n & 7)),
// kRImgBytes each, 128-byte aligned
constexpr int kRImgBytes = 3 * 2 * kD * 128;  // 98,304
constexpr int kRKImgOff = kMetaCOff + kMetaCFloats, kRVImgOff = kRKImgOff + kRImgBytes / 4;
constexpr int kParamFloats = kRVImgOff + kRImgBytes / 4;
static_assert(kRKImgOff % 32 == 0 && kParamFloats % 32 == 0, "128-byte aligned parameter regions");
// one split partial: m (log2 units), l, then acc[D]; padded to 132 floats (528 B, 16 B aligned)
constexpr int kPartFloats = kD + 4;
constexpr float kLog2e = 1.4426950408889634f;

// Device view of one layer of a cache.
struct LayerView {
  uint8_t* int2;          // [n_int2][hkv][kBlockBytes]
  uint8_t* bf16;          // [n_bf16][hkv][kBf16BlockBytes]
  const float* params;    // [hkv][kParamFloats]
  const float* next_params;   // the next layer's parameters (prefetched into L2 by the prologue), or null
  int n_int2, n_bf16, hkv, hq, sink, recent, v_explicit;
  int meta_u8;            // OSCAR_META_U8 pool: 8-bit (mn8, mx8) metadata, 4608-byte INT2 blocks
  int meta_cb;            // OSCAR_META_CB pool: codebook levels, fp16 (range, zero) metadata
  int blk_bytes;          // INT2 block bytes: kBlockBytes or kBlockBytesU8
  int* status;            // device status word
  int layer;              // layer index (timeline records only)
  unsigned long long* timeline;   // optional kernel timeline (see oscar_trace_timeline), or null
  int timeline_cap;       // records available in timeline
};

__device__ __forceinline__ void flag(int* status, int bits) { atomicOr(status, bits); }

// NaN or infinity (false for every finite float)
__device__ __forceinline__ bool nonfinite(float x) { return !(fabsf(x) <= 3.402823466e38f); }
// one of the two bf16 values of a 32-bit word is a NaN or an infinity (exponent bits all set)
__device__ __forceinline__ bool bf16x2_nonfinite(uint32_t w) {
  return ((w & 0x7F80u) == 0x7F80u) || ((w & 0x7F800000u) == 0x7F800000u);
}
// fp16 metadata that would not fit: |x| beyond the largest finite fp16 (or NaN)
__device__ __forceinline__ bool fp16_saturates(float x) { return !(fabsf(x) <= 65504.f); }

__device__ __forceinline__ const uint8_t* int2_block(const LayerView& lv, int page, int head) {
  return lv.int2 + ((size_t)page * lv.hkv + head) * lv.blk_bytes;
}
__device__ __forceinline__ uint8_t* int2_block_w(const LayerView& lv, int page, int head) {
  return lv.int2 + ((size_t)page * lv.hkv + head) * lv.blk_bytes;
}
// Grid constants {T, D, E, 0} of (kv head h, kind, group G) of the compact format.
__device__ __forceinline__ const float* meta_consts(const LayerView& lv, int h, int kind) {
  return lv.params + (size_t)h * kParamFloats + kMetaCOff + kind * 8;
}

// Codebook constants {k_0..k_3, theta_0..theta_2, 0} of (kv head h, kind).
__device__ __forceinline__ const float* cb_consts(const LayerView& lv, int h, int kind) {
  return lv.params + (size_t)h * kParamFloats + kCbOff + kind * 8;
}
// Codebook format, write side: the code of t = (y - zero') / range' (0 .. 3, ties to the lower level).
__device__ __forceinline__ float cb_code(float t, const float* cb) {
  return (float)((t > cb[4]) + (t > cb[5]) + (t > cb[6]));
}

// Compact format, write side: the group's grid indices from its clipped min / max, and the
// dequantisation parameters the codes are computed with. Every operation rounds as written: the
// quotients with __fadd_rn / __fdiv_rn, zero' = fma(mn8, D, -T), scale' = (mx8 - mn8) * E.
__device__ __forceinline__ void u8_quant_params(float mn, float mx, float T, float D, float E, unsigned& mn8,
                                                unsigned& mx8, float& scale, float& zero) {
  mn8 = mx8 = 0u;
  if (D > 0.f) {
    const float lo = floorf(__fdiv_rn(__fadd_rn(mn, T), D));
    const float hi = ceilf(__fdiv_rn(__fadd_rn(mx, T), D));
    mn8 = (unsigned)fminf(fmaxf(lo, 0.f), 255.f);
    mx8 = (unsigned)fminf(fmaxf(hi, 0.f), 255.f);
  }
  scale = __fmul_rn((float)(mx8 - mn8), E);
  zero = __fmaf_rn((float)mn8, D, -T);
}
// Compact format, read side: (scale', zero') of one group from its two index bytes.
__device__ __forceinline__ float2 u8_scale_zero(unsigned mn8, unsigned mx8, float T, float D, float E) {
  return make_float2(__fmul_rn((float)(int)(mx8 - mn8), E), __fmaf_rn((float)mn8, D, -T));
}
__device__ __forceinline__ __nv_bfloat16* bf16_row(const LayerView& lv, int page, int head, int kind, int row) {
  return reinterpret_cast<__nv_bfloat16*>(lv.bf16 + ((size_t)page * lv.hkv + head) * kBf16BlockBytes) +
         (size_t)kind * kP * kD + (size_t)row * kD;
}

// V codes are channel-major: channel c's 64 codes occupy the 16-byte slot c ^ ((c >> 4) & 7) of the V
// region (the swizzle puts channels 16 g + m, g = 0..7, in distinct banks). Row t's code sits in the
// slot's 32-bit word (t >> 1) & 3 at bit 16 (t & 1) + 4 (t >> 4) + 2 ((t >> 3) & 1): word w holds the rows
// t with t % 16 in {2w, 2w + 1, 2w + 8, 2w + 9}, even rows in its low half and each odd partner at the
// same position of the high half, code position 2 (t >> 4) + ((t >> 3) & 1). One masked word is then the
// fp16 pair of two consecutive rows, and word w gives a tensor-core lane t = w all its pairs of a page.
constexpr int kVChanBytes = kP / 4;            // 16
__device__ __forceinline__ int v_chan_off(int c) { return kVCodesOff + (c ^ ((c >> 4) & 7)) * kVChanBytes; }
__device__ __forceinline__ int v_word(int t) { return (t >> 1) & 3; }
__device__ __forceinline__ int v_bit(int t) { return 16 * (t & 1) + 4 * (t >> 4) + 2 * ((t >> 3) & 1); }

// Set the 2-bit V field of (channel c, row t) of a page block to `code`, leaving the other rows' bits:
// two atomics on the field's 32-bit word, so that writers of other rows of the same word may run at the
// same time.
__device__ __forceinline__ void v_set_code(uint8_t* blk, int c, int t, unsigned code) {
  unsigned* w = reinterpret_cast<unsigned*>(blk + v_chan_off(c) + 4 * v_word(t));
  const int sh = v_bit(t);
  atomicAnd(w, ~(3u << sh));
  if (code != 0u) atomicOr(w, code << sh);
}

// 7-bit bit reversal (d = 128).
__device__ __forceinline__ int bitrev7(int i) { return (int)(__brev((unsigned)i) >> 25); }

}  // namespace oscar
