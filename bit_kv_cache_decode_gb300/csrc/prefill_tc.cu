// Bulk prefill on the 5th-generation tensor cores (sm_103a): the write path's
// rotate, clip, quantise and pack over whole pages (MarkTechPost article
// "Together AI 开源 OSCAR…", section "服务系统：混合精度缓存布局": rotation,
// percentile clipping, per-token asymmetric INT2 over 64-channel groups, packed
// codes; news article "超越 TurboQuant…OSCAR…", section "OSCAR 的设计思路":
// prefill tokens land in the sink, the history and the recent window).
//
// Two kernels:
//  * k_prefill_bf16 copies the sink and recent rows of every request (bf16,
//    grid (request, kv head, K / V));
//  * k_prefill_tc quantises the history: one persistent CTA per SM walks a
//    contiguous share of the work items (kind, kv head, tile), a tile being
//    128 history rows of one request that start at a page-pair boundary (so a
//    tile owns its two pages' code and metadata bytes outright). Warp roles:
//    - warp 0 loads each tile's rows with two tensor-map copies (64 channels
//      each, 128-byte swizzle) into a 3-stage ring, and the B operand of the
//      (kind, head) when it changes: the rotation's three bf16 parts as a
//      prepared image (K, and V in explicit-V mode), or the identity (V in
//      V-absorbed mode, stored as it comes);
//    - warp 1 owns 512 TMEM columns (four 128-column accumulators) and issues
//      Y = X b1 + X b2 + X b3 (M = 128 rows, N = 128 channels, K = 16 per
//      instruction; 24 instructions a tile, 8 for the identity); every bf16
//      product is exact and the sum is accumulated in float32;
//    - warps 2..17 form two teams of eight that take alternate tiles: warp
//      (TMEM lane quarter q, group G) quantises the 32 rows x 64 channels it
//      reads from the accumulator: clip to +-tau, group min / max, the format's
//      scale and zero, codes (below), then writes K codes and all metadata to
//      the page rows and V codes, which are channel-major, through a
//      transposing buffer in shared memory, one 16-byte channel slot a thread.
//  Codes: code = clamp(rint(fl((y - zero) / scale)), 0, 3) with round half to
//  even (the codebook format: the level of fl((y - zero) / range)), as the
//  single-row quantiser computes them. The quotient is obtained without a
//  division: exactly, from a two-float reciprocal, where the scale is an fp16
//  value; within 3 ulp for the compact format, whose rare near-boundary values
//  are settled exactly (see quantise_group).
#include <algorithm>
#include <cuda.h>

#include "kernels.cuh"
#include "rotate.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"
#include "timeline.cuh"

namespace oscar {
namespace {

constexpr int kTile = 2 * kP;                          // history rows per tile
constexpr int kStages = 3;
constexpr int kBoxBytes = kTile * 128;                 // 16 KB: 128 rows x 64 bf16 channels
constexpr int kStageBytes = 2 * kBoxBytes;             // 32 KB
constexpr int kYBufs = 4;                              // TMEM accumulators of 128 columns
constexpr int kTeams = 2, kTeamThreads = 256;
constexpr int kThreads = 64 + kTeams * kTeamThreads;   // 576: loader, MMA, two epilogue teams
constexpr int kCsStride = kTile + 4;                   // transposing buffer: 132 bytes per channel quad
constexpr int kCsBytes = (kD / 4) * kCsStride;         // 4,224
constexpr int kOffStage = 0;
constexpr int kOffB = kOffStage + kStages * kStageBytes;          // 98,304
constexpr int kOffCs = kOffB + kRImgBytes;                         // 196,608: [team][kCsBytes]
constexpr int kOffBar = kOffCs + kTeams * kCsBytes;               // 205,056
// barriers: full[3], empty[3], b_full, b_free, y_full[4], y_empty[4], fin; then the TMEM address
constexpr int kBarFull = 0, kBarEmpty = kStages, kBarBFull = 2 * kStages, kBarBFree = kBarBFull + 1,
              kBarYFull = kBarBFree + 1, kBarYEmpty = kBarYFull + kYBufs, kBarFin = kBarYEmpty + kYBufs,
              kNumBars = kBarFin + 1;
constexpr int kPrefSmem = kOffBar + kNumBars * 8 + 8 + 1024;       // + alignment slack
constexpr uint32_t kIdescBf16 = idesc_f16(128, 128) | (1u << 7) | (1u << 10);   // A, B bf16
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

static_assert(kPrefSmem <= 232448, "shared memory");

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
// named barrier of one epilogue team (ids 1, 2): plain, and with an AND over the team's predicates
// (bar.sync and bar.red are warp-aligned: each warp reconverges first)
__device__ __forceinline__ void team_sync(int team) {
  __syncwarp();
  asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(kTeamThreads) : "memory");
}
__device__ __forceinline__ bool team_and(int team, bool p) {
  uint32_t r;
  __syncwarp();
  asm volatile(
      "{\n.reg .pred a, b;\nsetp.ne.u32 a, %1, 0;\nbar.red.and.pred b, %2, %3, a;\nselp.u32 %0, 1, 0, b;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)p), "r"(1 + team), "r"(kTeamThreads)
      : "memory");
  return r != 0;
}

// history rows of request r and its tiles
__device__ __forceinline__ int hist_rows(const LayerView& lv, const int* cu, int r) {
  return max(0, cu[r + 1] - cu[r] - lv.sink - lv.recent);
}
__device__ __forceinline__ int req_tiles(const LayerView& lv, const int* cu, int r) {
  return (hist_rows(lv, cu, r) + kTile - 1) / kTile;
}

// Work item n = p * T + t: pair p = kind * hkv + head, tile t of the batch's T tiles in request order
// (request r, its tile j). Walks are warp-uniform.
struct Walk {
  int p, t, r, j;
};
// the batch's tiles, by a whole warp
__device__ int batch_tiles(const LayerView& lv, const int* cu, int B) {
  int s = 0;
  for (int r = (threadIdx.x & 31); r < B; r += 32) s += req_tiles(lv, cu, r);
  return __reduce_add_sync(0xffffffffu, s);
}
// position a walk at item n, by a whole warp
__device__ void walk_seek(Walk& w, long long n, int T, const LayerView& lv, const int* cu, int B) {
  const int lane = threadIdx.x & 31;
  w.p = (int)(n / T);
  w.t = (int)(n % T);
  int left = w.t;
  w.r = B;
  w.j = 0;
  for (int r0 = 0; r0 < B; r0 += 32) {
    const int nt = r0 + lane < B ? req_tiles(lv, cu, r0 + lane) : 0;
    int incl = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, incl > left);
    if (hit != 0u) {
      const int l = __ffs(hit) - 1;
      w.r = r0 + l;
      w.j = left - __shfl_sync(0xffffffffu, incl - nt, l);
      return;
    }
    left -= __shfl_sync(0xffffffffu, incl, 31);
  }
}
__device__ __forceinline__ void walk_next(Walk& w, int T, const LayerView& lv, const int* cu, int B) {
  ++w.j;
  if (++w.t == T) {
    ++w.p;
    w.t = 0;
    w.r = 0;
    w.j = 0;
  }
  while (w.r < B && w.j >= req_tiles(lv, cu, w.r)) {
    w.j = 0;
    ++w.r;
  }
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
    // the quotient is monotone in y: unless the group's largest one rounds past 3, no code needs the
    // upper clamp (it takes fp16 rounding of a narrow group's scale and zero to get there)
    const float dmax = __fsub_rn(mx, zq);
    const bool hi_clamp = __fmaf_rn(dmax, rh, __fmul_rn(dmax, rl)) >= 3.5f;
    const bool any_hi = __any_sync(0xffffffffu, hi_clamp);
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
          if (any_hi) {
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

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1)
    k_prefill_tc(LayerView lv, const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                 const int* __restrict__ cu_seqlens, int B, const int* __restrict__ hist_pt, int max_hist_pages) {
  TimelineSpan timeline_span(lv, kTlPrefill);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sb = smem_addr(smem);
  auto bar = [&](int i) { return sb + (uint32_t)kOffBar + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + kNumBars * 8);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init_n(bar(kBarFull + s), 1);
      mbar_init_n(bar(kBarEmpty + s), 1);
    }
    mbar_init_n(bar(kBarBFull), 1);
    mbar_init_n(bar(kBarBFree), 1);
    for (int b = 0; b < kYBufs; ++b) {
      mbar_init_n(bar(kBarYFull + b), 1);
      mbar_init_n(bar(kBarYEmpty + b), 8);     // one arrival per warp of the team
    }
    mbar_init_n(bar(kBarFin), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kYBufs * 128)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int T = batch_tiles(lv, cu_seqlens, B);
  const long long N = 2LL * lv.hkv * T;
  const long long n0 = N * blockIdx.x / gridDim.x, n1 = N * (blockIdx.x + 1) / gridDim.x;
  const int cnt = (int)(n1 - n0);
  bool ok = true;

  if (cnt > 0 && warp == 0) {
    // ---- loader: the B operand when the (kind, head) changes, then each tile's rows ----
    const uint64_t pol = l2_evict_first();
    Walk w;
    walk_seek(w, n0, T, lv, cu_seqlens, B);
    int cur_p = -1, nsw = 0, i = 0;
    for (; i < cnt; ++i) {
      const int h = w.p % lv.hkv, kind = w.p / lv.hkv;
      if (w.p != cur_p) {
        if (nsw > 0) {                           // the previous operand's MMAs have completed
          bool good = lane == 0 ? mbar_wait(bar(kBarBFree), (nsw - 1) & 1) : true;
          if (!__shfl_sync(0xffffffffu, good, 0)) {
            ok = false;
            break;
          }
        }
        if (kind == OSCAR_KIND_K || lv.v_explicit) {
          if (lane == 0) {
            const uint8_t* img = reinterpret_cast<const uint8_t*>(
                lv.params + (size_t)h * kParamFloats + (kind == OSCAR_KIND_K ? kRKImgOff : kRVImgOff));
            mbar_expect_tx(bar(kBarBFull), kRImgBytes);
            for (int c = 0; c < 3; ++c) bulk_copy(sb + kOffB + c * 32768, img + c * 32768, 32768, bar(kBarBFull));
          }
        } else {                                 // the identity: V stored as it comes
          uint4* z = reinterpret_cast<uint4*>(smem + kOffB);
          for (int x = lane; x < 32768 / 16; x += 32) z[x] = make_uint4(0u, 0u, 0u, 0u);
          __syncwarp();
          for (int n = lane; n < kD; n += 32) {
            const int off = (n >> 6) * 16384 + n * 128 + ((((n & 63) >> 3) ^ (n & 7)) << 4) + (n & 7) * 2;
            *reinterpret_cast<uint16_t*>(smem + kOffB + off) = 0x3F80;   // bf16 1.0
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarBFull));
        }
        cur_p = w.p;
        ++nsw;
      }
      const int s = i % kStages;
      bool good = true;
      if (lane == 0) {
        good = mbar_wait(bar(kBarEmpty + s), ((i / kStages) & 1) ^ 1);
        if (good) {
          const CUtensorMap* map = kind == OSCAR_KIND_K ? &map_k : &map_v;
          const int tok = cu_seqlens[w.r] + lv.sink + kTile * w.j;
          const uint32_t dst = sb + kOffStage + s * kStageBytes;
          mbar_expect_tx(bar(kBarFull + s), kStageBytes);
          tma_load_3d(dst, map, 0, h, tok, bar(kBarFull + s), pol);
          tma_load_3d(dst + kBoxBytes, map, 64, h, tok, bar(kBarFull + s), pol);
        }
      }
      if (!__shfl_sync(0xffffffffu, good, 0)) {
        ok = false;
        break;
      }
      walk_next(w, T, lv, cu_seqlens, B);
    }
    // every copy this warp issued lands before the CTA may exit
    if (lane == 0) {
      for (int k = max(0, i - kStages); k < i; ++k)
        if (!mbar_wait(bar(kBarFull + k % kStages), (k / kStages) & 1)) ok = false;
      if (nsw > 0 && !mbar_wait(bar(kBarBFull), (nsw - 1) & 1)) ok = false;
    }
  } else if (cnt > 0 && warp == 1) {
    // ---- MMA issue: Y[b] = X (b1 + b2 + b3), or X I ----
    Walk w;
    walk_seek(w, n0, T, lv, cu_seqlens, B);
    int cur_p = -1, nsw = 0, parts = 3;
    for (int i = 0; i < cnt; ++i) {
      const int s = i % kStages, b = i % kYBufs;
      bool good = true;
      if (w.p != cur_p) {
        if (lane == 0) good = mbar_wait(bar(kBarBFull), nsw & 1);
        parts = (w.p / lv.hkv == OSCAR_KIND_K || lv.v_explicit) ? 3 : 1;
        cur_p = w.p;
        ++nsw;
      }
      if (lane == 0 && good)
        good = mbar_wait(bar(kBarFull + s), (i / kStages) & 1) &&
               mbar_wait(bar(kBarYEmpty + b), ((i / kYBufs) & 1) ^ 1);
      if (!__shfl_sync(0xffffffffu, good, 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
      walk_next(w, T, lv, cu_seqlens, B);
      if (lane == 0) {
        const uint32_t a0 = sb + kOffStage + s * kStageBytes, b0 = sb + kOffB, d = tmem + 128u * b;
        for (int p = 0; p < parts; ++p)
#pragma unroll
          for (int kh = 0; kh < 2; ++kh)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma(d, desc_sw128(a0 + kh * kBoxBytes + 32 * ks), desc_sw128(b0 + p * 32768 + kh * 16384 + 32 * ks),
                   kIdescBf16, (p | kh | ks) != 0);
        umma_commit(bar(kBarEmpty + s));         // the stage is free once these MMAs complete
        umma_commit(bar(kBarYFull + b));
        if (i == cnt - 1 || w.p != cur_p) umma_commit(bar(kBarBFree));
      }
      __syncwarp();
    }
    if (lane == 0) {                             // every MMA has completed before TMEM is released
      umma_commit(bar(kBarFin));
      if (!mbar_wait(bar(kBarFin), 0)) ok = false;
    }
  } else if (cnt > 0) {
    // ---- epilogue teams: warp (quarter q, group G) quantises rows 32 q .. 32 q + 31, channels 64 G .. ----
    const int e = warp - 2, team = e >> 3, G = (e >> 2) & 1, q = warp & 3;
    const int row = 32 * q + lane;
    const int u = (e & 7) * 32 + lane;           // index within the team (V transpose)
    uint8_t* cs = smem + kOffCs + team * kCsBytes;
    Walk w;
    walk_seek(w, n0, T, lv, cu_seqlens, B);
    for (int i = 0; i < cnt; ++i) {
      if ((i & 1) == team) {
        const int b = i % kYBufs;
        // the team decides together (it also orders this tile's transposing-buffer writes after the
        // previous tile's reads)
        if (!team_and(team, mbar_wait(bar(kBarYFull + b), (i / kYBufs) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int h = w.p % lv.hkv, kind = w.p / lv.hkv, r = w.r, h0 = kTile * w.j;
        const int hn = min(kTile, hist_rows(lv, cu_seqlens, r) - h0);
        const bool row_ok = row < hn;
        const float* prm = lv.params + (size_t)h * kParamFloats;
        uint32_t wd[4], meta;
        bool nf, sat;
        quantise_group<FMT>(tmem + ((uint32_t)(32 * q) << 16) + 128u * b + 64u * G, prm, kind, G, wd, meta, nf,
                            sat);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarYEmpty + b));   // the accumulator is free for the MMA
        // this row's page; a bad page id skips the row (and is flagged)
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
            *reinterpret_cast<uint4*>(blk + kKCodesOff + prow * (kD / 4) + 16 * G) =
                make_uint4(wd[0], wd[1], wd[2], wd[3]);
          if constexpr (FMT == kFmtU8)
            *reinterpret_cast<uint16_t*>(blk + (kind == OSCAR_KIND_K ? kKMetaOff : kVMetaOffU8) + prow * (kNG * 2) +
                                         2 * G) = (uint16_t)meta;
          else
            *reinterpret_cast<uint32_t*>(blk + (kind == OSCAR_KIND_K ? kKMetaOff : kVMetaOff) + prow * (kNG * 4) +
                                         4 * G) = meta;
        }
        if (kind == OSCAR_KIND_V) {
          // codes by channel quad: byte (quad, row) = the codes of channels 4 quad .. 4 quad + 3 of the row
          // (zero past the tile's rows); then thread u writes channel u % 128's slot of page u / 128
#pragma unroll
          for (int k = 0; k < 16; ++k)
            cs[(16 * G + k) * kCsStride + row] = row_ok ? (uint8_t)(wd[k >> 2] >> (8 * (k & 3))) : (uint8_t)0;
          team_sync(team);
          const int c = u & (kD - 1), pg = u >> 7;
          if (pg * kP < hn) {
            const int hpg = h0 / kP + pg;
            const int pid = hpg < max_hist_pages ? hist_pt[(size_t)r * max_hist_pages + hpg] : -1;
            if (pid >= 0 && pid < lv.n_int2) {   // a bad id was flagged by its rows
              const uint8_t* src = cs + (c >> 2) * kCsStride + kP * pg;
              const int sh = 2 * (c & 3);
              uint32_t wv[4] = {0u, 0u, 0u, 0u};
              // rows 4j .. 4j + 3: rows 4j, 4j + 1 in word (2j) & 3 at bits p and p + 16, rows 4j + 2, 4j + 3
              // in the next word, p = 4 (j / 4) + 2 ((j / 2) & 1)
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const uint32_t x = (*reinterpret_cast<const uint32_t*>(src + 4 * j) >> sh) & 0x03030303u;
                const int wq = (2 * j) & 3, p = 4 * (j >> 2) + 2 * ((j >> 1) & 1);
                wv[wq] += __byte_perm(x, 0u, 0x4140) << p;
                wv[wq + 1] += __byte_perm(x, 0u, 0x4342) << p;
              }
              *reinterpret_cast<uint4*>(int2_block_w(lv, pid, h) + v_chan_off(c)) =
                  make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
          }
        }
      }
      walk_next(w, T, lv, cu_seqlens, B);
    }
  }
  if (!ok && lane == 0) flag(lv.status, OSCAR_STATUS_TIMEOUT);
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kYBufs * 128) : "memory");
  }
}

// Sink and recent rows of request r, kv head h, one kind: bf16 copies, one warp per row.
__global__ void __launch_bounds__(128) k_prefill_bf16(LayerView lv, const __nv_bfloat16* __restrict__ k,
                                                      const __nv_bfloat16* __restrict__ v,
                                                      const int* __restrict__ cu_seqlens, const int* __restrict__ bf16_pt) {
  pdl_launch_dependents();                       // the history kernel touches other memory: let it start
  const int r = blockIdx.x, h = blockIdx.y, kind = blockIdx.z;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = cu_seqlens[r + 1] - cu_seqlens[r];
  const int bf16_per_req = (lv.sink + lv.recent) / kP;
  const __nv_bfloat16* src = kind == OSCAR_KIND_K ? k : v;
  const int nsink = min(L, lv.sink), rec0 = max(lv.sink, L - lv.recent);
  const int n = nsink + max(0, L - rec0);
  for (int i = w; i < n; i += 4) {
    const int pos = i < nsink ? i : rec0 + (i - nsink);
    int page, row;
    if (pos < lv.sink) {
      page = bf16_pt[r * bf16_per_req + pos / kP];
      row = pos % kP;
    } else {
      const int slot = (pos - lv.sink) % lv.recent;
      page = bf16_pt[r * bf16_per_req + lv.sink / kP + slot / kP];
      row = slot % kP;
    }
    if (page < 0 || page >= lv.n_bf16) {
      if (lane == 0) flag(lv.status, OSCAR_STATUS_BAD_PAGE);
      continue;
    }
    const uint2 x = reinterpret_cast<const uint2*>(src + (((size_t)cu_seqlens[r] + pos) * lv.hkv + h) * kD)[lane];
    if (__any_sync(0xffffffffu, bf16x2_nonfinite(x.x) || bf16x2_nonfinite(x.y)) && lane == 0)
      flag(lv.status, OSCAR_STATUS_NONFINITE);
    reinterpret_cast<uint2*>(bf16_row(lv, page, h, kind, row))[lane] = x;
  }
}

}  // namespace

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
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
// [total tokens][hkv][128] bf16 as a 3-D tensor (channel, head, token); boxes of 64 channels x 1 head x 128
// tokens land 128-byte swizzled; tokens past the end read as zero
bool row_map(CUtensorMap* map, const void* base, int hkv, int total) {
  EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)hkv, (cuuint64_t)total};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)hkv * kD * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kTile};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

int launch_prefill(const LayerView& lv, int B, const void* k, const void* v, const int* cu_seqlens, int total,
                   const int* hist_pt, int max_hist_pages, const int* bf16_pt, cudaStream_t st) {
  if (total == 0 || B == 0) return OSCAR_OK;
  const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(k);
  const __nv_bfloat16* vb = static_cast<const __nv_bfloat16*>(v);
  k_prefill_bf16<<<dim3(B, lv.hkv, 2), 128, 0, st>>>(lv, kb, vb, cu_seqlens, bf16_pt);
  CUtensorMap map_k, map_v;
  if (!row_map(&map_k, k, lv.hkv, total) || !row_map(&map_v, v, lv.hkv, total)) return OSCAR_ERR_CUDA;
  // one CTA per SM, each walking a contiguous share of the (kind, head, tile) items
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long items_max = 2LL * lv.hkv * ((long long)total / kTile + B);
  const int grid = (int)std::max(1LL, std::min((long long)sms, items_max));
  // launched as a programmatic dependent of the sink / recent copy, which it runs beside (neither waits
  // for the other; later work on the stream waits for both)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kPrefSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (lv.meta_u8)
    e = cudaLaunchKernelEx(&cfg, k_prefill_tc<kFmtU8>, lv, map_k, map_v, cu_seqlens, B, hist_pt, max_hist_pages);
  else if (lv.meta_cb)
    e = cudaLaunchKernelEx(&cfg, k_prefill_tc<kFmtCB>, lv, map_k, map_v, cu_seqlens, B, hist_pt, max_hist_pages);
  else
    e = cudaLaunchKernelEx(&cfg, k_prefill_tc<kFmtF16>, lv, map_k, map_v, cu_seqlens, B, hist_pt, max_hist_pages);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int configure_prefill_kernel() {
  const bool ok =
      cudaFuncSetAttribute(k_prefill_tc<kFmtF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrefSmem) ==
          cudaSuccess &&
      cudaFuncSetAttribute(k_prefill_tc<kFmtU8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrefSmem) ==
          cudaSuccess &&
      cudaFuncSetAttribute(k_prefill_tc<kFmtCB>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrefSmem) ==
          cudaSuccess;
  return ok ? OSCAR_OK : OSCAR_ERR_CUDA;
}

}  // namespace oscar
