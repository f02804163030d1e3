// Shared pieces of the tensor-core write-path kernels (the bulk prefill and the fused projection
// prefill): 128-byte-swizzled operand descriptors and tensor-map loads, the quantiser of one row's
// 64-channel group read from tensor memory, and the store of a 128-row history tile's codes and
// metadata (MarkTechPost article "Together AI 开源 OSCAR…", section "服务系统：混合精度缓存布局":
// clip to per-channel thresholds, per-token asymmetric INT2 over 64-channel groups, packed codes).
#pragma once

#include <cuda.h>

#include "kernels.cuh"
#include "rotate.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace oscar {
namespace qtile {

// the driver's tensor-map encoder, found once through the runtime (no link against the driver library)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
inline EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

constexpr int kRows = 2 * kP;                          // rows of a history tile (two pages)
constexpr int kBoxBytes = kRows * 128;                 // 16 KB: 128 rows x 64 bf16 channels, swizzled
constexpr int kCsStride = kRows + 4;                   // transposing buffer: 132 bytes per channel quad
constexpr int kCsBytes = (kD / 4) * kCsStride;         // 4,224
constexpr int kTeamThreads = 256;                      // an epilogue team: 8 warps, 4 lane quarters x 2 groups
constexpr uint32_t kIdescBf16 = idesc_f16(128, 128) | (1u << 7) | (1u << 10);   // A, B bf16, M 128, N 128
constexpr float kMagic = 12582912.f;                   // 1.5 * 2^23: x + kMagic rounds x to an integer
constexpr float kNearHalf = 0.5f - 0x1p-20f;           // |q - rint(q)| above this: the division decides

// sum over m < 16 of (bits of kMagic) << 2m, modulo 2^32: packing (bits of q + kMagic) << 2m leaves the
// codes plus this constant
constexpr uint32_t magic_pack() {
  uint32_t s = 0u;
  for (int m = 0; m < 16; ++m) s += 0x4B400000u << (2 * m);
  return s;
}
constexpr uint32_t kMagicPack = magic_pack();


// UMMA shared-memory descriptor, K-major with the 128-byte swizzle: 8-row blocks 1024 bytes apart
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// named barrier `id` over `n` threads: plain, and with an AND over their predicates (bar.sync and
// bar.red are warp-aligned: each warp reconverges first)
__device__ __forceinline__ void named_sync(int id, int n) {
  __syncwarp();
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ bool named_and(int id, int n, bool p) {
  uint32_t r;
  __syncwarp();
  asm volatile(
      "{\n.reg .pred a, b;\nsetp.ne.u32 a, %1, 0;\nbar.red.and.pred b, %2, %3, a;\nselp.u32 %0, 1, 0, b;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)p), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
// byte offset of element (n, k) in a B operand of 128 rows n x 128 channels k, K-major, 128-byte swizzle
__device__ __forceinline__ int sw128_offset(int n, int k) {
  return (k >> 6) * kBoxBytes + n * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) + (k & 7) * 2;
}

// Quantise one row's group of 64 rotated values, which sit in TMEM at `ty` (this thread's lane, 64
// columns): clip (the clipped values go back to TMEM), group min / max, the format's scale and zero, codes;
// wd[q4] holds channels 16 q4 + m at bits 2m.
template <int FMT>
__device__ __forceinline__ void quantise_group(uint32_t ty, const float* prm, int kind, int G, uint32_t (&wd)[4],
                                               uint32_t& meta, bool& nf, bool& sat) {
  const float4* tau4 = reinterpret_cast<const float4*>(prm + (kind == OSCAR_KIND_K ? kTauKOff : kTauVOff) + 64 * G);
  float mn = INFINITY, mx = -INFINITY;
  float nfa = 0.f;                               // stays 0 unless a value is NaN or infinite (x * 0 is NaN)
#pragma unroll 1
  for (int hf = 0; hf < 2; ++hf) {
    float y[32];
    tmem_ld32(ty + 32 * hf, y);
#pragma unroll
    for (int i4 = 0; i4 < 8; ++i4) {
      const float4 t = __ldg(tau4 + 8 * hf + i4);
      float* a = y + 4 * i4;
      nfa = __fmaf_rn(a[0], 0.f, __fmaf_rn(a[1], 0.f, __fmaf_rn(a[2], 0.f, __fmaf_rn(a[3], 0.f, nfa))));
      a[0] = fminf(fmaxf(a[0], -t.x), t.x);
      a[1] = fminf(fmaxf(a[1], -t.y), t.y);
      a[2] = fminf(fmaxf(a[2], -t.z), t.z);
      a[3] = fminf(fmaxf(a[3], -t.w), t.w);
      mn = min3f(min3f(mn, a[0], a[1]), a[2], a[3]);
      mx = max3f(max3f(mx, a[0], a[1]), a[2], a[3]);
    }
    tmem_st32(ty + 32 * hf, y);
  }
  nf = nfa != 0.f;
  float sq, zq;
  sat = false;
  if constexpr (FMT == kFmtU8) {
    const float* mc = prm + kMetaCOff + kind * 8 + 4 * G;
    unsigned mn8, mx8;
    u8_quant_params(mn, mx, mc[0], mc[1], mc[2], mn8, mx8, sq, zq);
    meta = mn8 | (mx8 << 8);
  } else {                                       // fp16 (scale, zero), or (range, zero) with a codebook
    const float diff = __fsub_rn(mx, mn);
    const float scale = FMT == kFmtCB ? diff : __fdiv_rn(diff, 3.0f);
    sat = fp16_saturates(scale) || fp16_saturates(mn);
    const __half2 sz = __halves2half2(__float2half_rn(sat_fp16(scale)), __float2half_rn(sat_fp16(mn)));
    sq = __low2float(sz);
    zq = __high2float(sz);
    meta = *reinterpret_cast<const uint32_t*>(&sz);
  }
  if constexpr (FMT != kFmtU8) {
    // scale is an fp16 value (at most 11 significant bits). With 1 / scale as rh + rl (rh = fl(1 / scale),
    // rl = fl((1 - scale rh) rh), the residual exact), fl(d rh + fl(d rl)) lies within 2^-46 (relative) of
    // d / scale, while d / scale (a 24-bit over an 11-bit number) is never within 2^-36 of a float32
    // rounding midpoint: it is the correctly rounded quotient fl(d / scale), exactly as the division gives.
    float rh = 0.f, rl = 0.f;
    if (sq != 0.f) {
      rh = __frcp_rn(sq);
      rl = __fmul_rn(__fmaf_rn(-sq, rh, 1.f), rh);
    }
    const float rh4 = __fmul_rn(rh, 0.25f), rl4 = __fmul_rn(rl, 0.25f);
    const float* cbc = prm + kCbOff + kind * 8;
    // the quotient is monotone in y: unless the group's smallest one rounds below 0 or its largest past
    // 3 (it takes fp16 rounding of a narrow group's scale and zero to get there), no code needs a clamp,
    // and the codes come from packed pairs of adjacent values (no saturating form exists for those)
    const float dmax = __fsub_rn(mx, zq), dmin = __fsub_rn(mn, zq);
    const bool hi_clamp = __fmaf_rn(dmax, rh, __fmul_rn(dmax, rl)) >= 3.5f;
    const bool lo_clamp = __fmaf_rn(dmin, rh, __fmul_rn(dmin, rl)) < -0.5f;
    const bool any_hi = __any_sync(0xffffffffu, hi_clamp);
    const bool all_in = !__any_sync(0xffffffffu, hi_clamp || lo_clamp);
    const float2 nzq2 = make_float2(-zq, -zq), rh2 = make_float2(rh, rh), rl2 = make_float2(rl, rl),
                 mg2 = make_float2(kMagic, kMagic);
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {
      float y[32];
      tmem_ld32(ty + 32 * hf, y);
      uint32_t w2[2];
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {
        uint32_t acc = 0u;
        if constexpr (FMT == kFmtCB) {
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            const float d = __fsub_rn(y[16 * q2 + m], zq);
            const float c = sq != 0.f ? cb_code(__fmaf_rn(d, rh, __fmul_rn(d, rl)), cbc) : 0.f;
            acc |= ((uint32_t)c) << (2 * m);
          }
          w2[q2] = acc;
        } else {
          // q/4 = sat(q / 4) (the scaling by 4 is exact), t = 4 (q/4) + kMagic rounds half to even;
          // min(t, kMagic + 3) clamps the code where a group needs it
          if (FMT == kFmtF16 && all_in) {
            // every quotient in [-0.5, 3.5): t = q + kMagic needs no clamp (-0.5 rounds to -0, code 0)
#pragma unroll
            for (int m = 0; m < 16; m += 2) {
              const float2 dd = __fadd2_rn(make_float2(y[16 * q2 + m], y[16 * q2 + m + 1]), nzq2);
              const float2 t = __fadd2_rn(__ffma2_rn(dd, rh2, __fmul2_rn(dd, rl2)), mg2);
              acc += __float_as_uint(t.x) << (2 * m);
              acc += __float_as_uint(t.y) << (2 * m + 2);
            }
          } else if (any_hi) {
#pragma unroll
            for (int m = 0; m < 16; ++m) {
              const float q4 = __saturatef(__fmaf_rn(__fsub_rn(y[16 * q2 + m], zq), rh4,
                                                     __fmul_rn(__fsub_rn(y[16 * q2 + m], zq), rl4)));
              acc += __float_as_uint(fminf(__fmaf_rn(q4, 4.f, kMagic), kMagic + 3.f)) << (2 * m);
            }
          } else {
#pragma unroll
            for (int m = 0; m < 16; ++m) {
              const float q4 = __saturatef(__fmaf_rn(__fsub_rn(y[16 * q2 + m], zq), rh4,
                                                     __fmul_rn(__fsub_rn(y[16 * q2 + m], zq), rl4)));
              acc += __float_as_uint(__fmaf_rn(q4, 4.f, kMagic)) << (2 * m);
            }
          }
          w2[q2] = acc - kMagicPack;
        }
      }
      if (hf == 0) {
        wd[0] = w2[0];
        wd[1] = w2[1];
      } else {
        wd[2] = w2[0];
        wd[3] = w2[1];
      }
    }
  } else {
    // compact format: scale = (mx8 - mn8) E has up to 24 significant bits. q = d fl(1 / scale) is within 3 ulp
    // of fl(d / scale), so rint can differ only within 2^-20 of a half-integer; a value that close keeps q if
    // q scale == d exactly (q is then the exact quotient; the exact ties of unrotated bf16 rows are such
    // values) and otherwise takes the IEEE division. q/4 = sat(q / 4) (the scaling by 4 is exact),
    // t = 4 (q/4) + kMagic rounds half to even, min(t, kMagic + 3) clamps the code.
    const float rs4 = sq != 0.f ? __fmul_rn(__frcp_rn(sq), 0.25f) : 0.f;
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {
      float y[32];
      tmem_ld32(ty + 32 * hf, y);
      bool near = false;
      uint32_t w2[2];
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {
        uint32_t acc = 0u;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float q4 = __saturatef(__fmul_rn(__fsub_rn(y[16 * q2 + m], zq), rs4));
          const float t = __fmaf_rn(q4, 4.f, kMagic);
          near |= fabsf(__fmaf_rn(q4, 4.f, -__fsub_rn(t, kMagic))) > kNearHalf;
          acc += __float_as_uint(fminf(t, kMagic + 3.f)) << (2 * m);
        }
        w2[q2] = acc - kMagicPack;
      }
      if (near) {                                // this lane only; the values are still in registers
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            const float d = __fsub_rn(y[16 * q2 + m], zq);
            const float q = __fmul_rn(__saturatef(__fmul_rn(d, rs4)), 4.f);
            const float c = __fsub_rn(__fadd_rn(q, kMagic), kMagic);
            if (fabsf(__fsub_rn(q, c)) > kNearHalf && __fmaf_rn(-q, sq, d) != 0.f) {
              const float ce = fminf(fmaxf(rintf(__fdiv_rn(d, sq)), 0.f), 3.f);
              w2[q2] = (w2[q2] & ~(3u << (2 * m))) | ((uint32_t)ce << (2 * m));
            }
          }
        }
      }
      if (hf == 0) {
        wd[0] = w2[0];
        wd[1] = w2[1];
      } else {
        wd[2] = w2[0];
        wd[3] = w2[1];
      }
    }
  }
}

// Store one history row's group G of a 128-row tile (history rows h0 .. h0 + hn - 1 of request r,
// kv head h, kind), thread `row` of the team's lane quarter and `u` its index in the team: the page
// lookup (a bad id skips the row and is flagged), K codes and all metadata straight to the page row,
// V codes (channel-major) through the team's transposing buffer `cs`, one 16-byte channel slot per
// thread; the team synchronises on named barrier `bar_id` (V only).
template <int FMT>
__device__ __forceinline__ void store_history_row(const LayerView& lv, const int* __restrict__ hist_pt,
                                                  int max_hist_pages, int r, int h, int kind, int h0, int hn,
                                                  int row, int G, int u, const uint32_t (&wd)[4], uint32_t meta,
                                                  bool nf, bool sat, uint8_t* cs, int bar_id) {
  const int lane = threadIdx.x & 31;
  const bool row_ok = row < hn;
  const int hp = (h0 + row) / kP, prow = (h0 + row) % kP;
  int page = -1;
  if (row_ok) {
    if (hp >= max_hist_pages) {
      flag(lv.status, OSCAR_STATUS_BAD_SEQLEN);
    } else {
      page = hist_pt[(size_t)r * max_hist_pages + hp];
      if (page < 0 || page >= lv.n_int2) {
        flag(lv.status, OSCAR_STATUS_BAD_PAGE);
        page = -1;
      }
    }
  }
  if (__any_sync(0xffffffffu, row_ok && nf) && lane == 0) flag(lv.status, OSCAR_STATUS_NONFINITE);
  if (__any_sync(0xffffffffu, row_ok && sat) && lane == 0) flag(lv.status, OSCAR_STATUS_SATURATED);
  if (page >= 0) {
    uint8_t* blk = int2_block_w(lv, page, h);
    if (kind == OSCAR_KIND_K)
      *reinterpret_cast<uint4*>(blk + kKCodesOff + prow * (kD / 4) + 16 * G) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    if constexpr (FMT == kFmtU8)
      *reinterpret_cast<uint16_t*>(blk + (kind == OSCAR_KIND_K ? kKMetaOff : kVMetaOffU8) + prow * (kNG * 2) + 2 * G) =
          (uint16_t)meta;
    else
      *reinterpret_cast<uint32_t*>(blk + (kind == OSCAR_KIND_K ? kKMetaOff : kVMetaOff) + prow * (kNG * 4) + 4 * G) =
          meta;
  }
  if (kind == OSCAR_KIND_V) {
    // codes by channel quad: byte (quad, row) = the codes of channels 4 quad .. 4 quad + 3 of the row (zero
    // past the tile's rows); then thread u writes channel u % 128's slot of page u / 128
#pragma unroll
    for (int k = 0; k < 16; ++k)
      cs[(16 * G + k) * kCsStride + row] = row_ok ? (uint8_t)(wd[k >> 2] >> (8 * (k & 3))) : (uint8_t)0;
    named_sync(bar_id, kTeamThreads);
    const int c = u & (kD - 1), pg = u >> 7;
    if (pg * kP < hn) {
      const int hpg = h0 / kP + pg;
      const int pid = hpg < max_hist_pages ? hist_pt[(size_t)r * max_hist_pages + hpg] : -1;
      if (pid >= 0 && pid < lv.n_int2) {         // a bad id was flagged by its rows
        const uint8_t* src = cs + (c >> 2) * kCsStride + kP * pg;
        const int sh = 2 * (c & 3);
        uint32_t wv[4] = {0u, 0u, 0u, 0u};
        // rows 4j .. 4j + 3: rows 4j, 4j + 1 in word (2j) & 3 at bits p and p + 16, rows 4j + 2, 4j + 3 in the
        // next word, p = 4 (j / 4) + 2 ((j / 2) & 1)
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t x = (*reinterpret_cast<const uint32_t*>(src + 4 * j) >> sh) & 0x03030303u;
          const int wq = (2 * j) & 3, p = 4 * (j >> 2) + 2 * ((j >> 1) & 1);
          wv[wq] += __byte_perm(x, 0u, 0x4140) << p;
          wv[wq + 1] += __byte_perm(x, 0u, 0x4342) << p;
        }
        *reinterpret_cast<uint4*>(int2_block_w(lv, pid, h) + v_chan_off(c)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
    }
  }
}

}  // namespace qtile
}  // namespace oscar
