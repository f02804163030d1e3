// Bulk prefill on the tensor cores (sm_103a): the write path's rotate, clip,
// quantise and pack over many tokens at once (MarkTechPost article "Together AI
// 开源 OSCAR…", section "服务系统：混合精度缓存布局": rotation, percentile
// clipping, per-token asymmetric INT2 over 64-channel groups, packed codes; the
// news article "超越 TurboQuant…OSCAR…", section "OSCAR 的设计思路": prefill
// tokens land in the sink, the history and the recent window).
//
// grid = (ceil(total / kPrefillTok), hkv, 2 kinds), block = 128 (4 warps). A CTA
// stages the (head, kind) rotation's fragments in shared memory once and walks
// kPrefillTok consecutive tokens of the flattened batch in 16-token tiles, one
// tile per warp at a time:
//  * the tile's 16 rows (bf16) are copied to shared memory, and each row is
//    classified (request by binary search in cu_seqlens; sink, history or
//    recent; destination page and row);
//  * sink and recent rows are copied as bf16;
//  * history rows are rotated as y = x R with R = U H P_br composed on the host:
//    A = x as fp16 (exact for bf16 values of normal fp16 range), B = R as
//    fp16 high + low parts, one fresh accumulator per 16-channel block (the
//    tensor cores' fp32 accumulation truncates), blocks added in rounding fp32;
//    V rows in V-absorbed mode are not rotated and take x itself;
//  * the quantiser works on the accumulator layout: lane (g, t) holds rows g
//    and g + 8, rotated channels 8 nt + 2t, +1 for n-tiles nt = 0..15 (group 0
//    = n-tiles 0-7). Every step is the same float32 operation, in the same
//    order, as the single-row quantiser: clip to +-tau, group min / max,
//    scale = (max - min) / 3, fp16 scale' and zero', code = rint((y - zero') /
//    scale') in [0, 3];
//  * codes go through shared memory and are packed into the page layout
//    (K token-major, V token-pair interleaved), with the fp16 metadata.
#include "kernels.cuh"
#include "rotate.cuh"
#include "tma.cuh"
#include "timeline.cuh"

namespace oscar {
namespace {

constexpr int kTileRows = 16;
constexpr int kXStride = kD + 8;                 // bf16 per staged row: 272 B, conflict-free fragment loads
constexpr int kPrefillWarps = 4;

__device__ __forceinline__ void mma16816_zero(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

__device__ __forceinline__ void mma16816_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// two bf16 (one 32-bit word) -> two fp16 packed
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

struct RowDest {
  int where;   // -1 nothing, 0 history, 1 bf16 (sink or recent)
  int page, row;
};

// Destination of flattened token index gtok (lane-local; invalid ids flag the status word).
__device__ __forceinline__ RowDest classify(const LayerView& lv, int gtok, int tok1, const int* cu_seqlens, int B,
                                            const int* hist_pt, int max_hist_pages, const int* bf16_pt) {
  RowDest d{-1, 0, 0};
  if (gtok >= tok1) return d;
  int lo = 0, hi = B;                            // request r: cu[r] <= gtok < cu[r+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu_seqlens[mid] <= gtok) lo = mid;
    else hi = mid;
  }
  const int r = lo, pos = gtok - cu_seqlens[r], L = cu_seqlens[r + 1] - cu_seqlens[r];
  const int bf16_per_req = (lv.sink + lv.recent) / kP;
  if (pos < lv.sink) {
    d.page = bf16_pt[r * bf16_per_req + pos / kP];
    d.row = pos % kP;
    d.where = 1;
  } else if (pos >= max(lv.sink, L - lv.recent)) {
    const int slot = (pos - lv.sink) % lv.recent;
    d.page = bf16_pt[r * bf16_per_req + lv.sink / kP + slot / kP];
    d.row = slot % kP;
    d.where = 1;
  } else {
    const int hh = pos - lv.sink;
    if (hh / kP >= max_hist_pages) {
      flag(lv.status, OSCAR_STATUS_BAD_SEQLEN);
      return d;
    }
    d.page = hist_pt[r * max_hist_pages + hh / kP];
    d.row = hh % kP;
    d.where = 0;
  }
  const int cap = d.where == 0 ? lv.n_int2 : lv.n_bf16;
  if (d.page < 0 || d.page >= cap) {
    flag(lv.status, OSCAR_STATUS_BAD_PAGE);
    d.where = -1;
  }
  return d;
}

// cp.async of 16 bytes global -> shared; src_bytes = 0 fills zeros (src is not read)
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Stage the 16 rows starting at flattened token `base` (bf16 [tok][hkv][128]) into xs.
__device__ __forceinline__ void stage_tile(__nv_bfloat16* xs, const __nv_bfloat16* src_all, int base, int tok1, int h,
                                           int hkv) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int c = lane + 32 * k, row = c >> 4, col8 = c & 15;
    const int tok = base + row;
    const bool ok = tok < tok1;
    const __nv_bfloat16* src = src_all + ((size_t)(ok ? tok : base) * hkv + h) * kD + 8 * col8;
    cp_async16(xs + row * kXStride + 8 * col8, src, ok ? 16 : 0);
  }
}

// 16 codes (one per byte, values 0..3) -> 32-bit word, code m at bits 2m
__device__ __forceinline__ uint32_t pack16(uint4 b) {
  auto pack4 = [](uint32_t x) -> uint32_t {
    return (x & 3u) | ((x >> 6) & 0xCu) | ((x >> 12) & 0x30u) | ((x >> 18) & 0xC0u);
  };
  return pack4(b.x) | (pack4(b.y) << 8) | (pack4(b.z) << 16) | (pack4(b.w) << 24);
}

// Rotate (or take) and quantise the staged 16-row tile xs, one 64-channel group (8 n-tiles) at a
// time; codes and fp16 metadata of every row go to codes_s [16][128] (one code per byte) and
// meta_s [16][2] (fp16 scale, zero per group). Rows whose bit is set in `checked` (the history rows)
// flag non-finite rotated values and saturated fp16 metadata in `status`.
__device__ __forceinline__ void quantize_tile(const uint32_t* frag_s, bool rotate, const __nv_bfloat16* xs,
                                              const float* tau_s, const float* mc, const float* cb,
                                              uint8_t* codes_s, uint32_t* meta_s, int* status, uint32_t checked) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  uint32_t a[8][4];
  if (rotate) {
    const uint32_t* x0 = reinterpret_cast<const uint32_t*>(xs + g * kXStride);
    const uint32_t* x8 = reinterpret_cast<const uint32_t*>(xs + (g + 8) * kXStride);
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      a[kb][0] = bf16x2_to_f16x2(x0[8 * kb + t]);          // row g, channels 16 kb + 2t, +1
      a[kb][1] = bf16x2_to_f16x2(x8[8 * kb + t]);          // row g + 8
      a[kb][2] = bf16x2_to_f16x2(x0[8 * kb + t + 4]);      // row g, channels 16 kb + 2t + 8, +9
      a[kb][3] = bf16x2_to_f16x2(x8[8 * kb + t + 4]);
    }
  }
#pragma unroll 1
  for (int G = 0; G < 2; ++G) {
    float acc[8][4];                                      // n-tiles 8 G .. 8 G + 7
    if (rotate) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int nt = 8 * G + j;
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          const uint4 b = *reinterpret_cast<const uint4*>(frag_s + ((kb * 16 + nt) * 32 + lane) * 4);
          float d[4];
          mma16816_zero(d, a[kb][0], a[kb][1], a[kb][2], a[kb][3], b.x, b.y);   // x R_hi
          mma16816_acc(d, a[kb][0], a[kb][1], a[kb][2], a[kb][3], b.z, b.w);    // + x R_lo
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[j][e] += d[e];
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int nt = 8 * G + j;
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(xs + g * kXStride + 8 * nt + 2 * t);
        const uint32_t w8 = *reinterpret_cast<const uint32_t*>(xs + (g + 8) * kXStride + 8 * nt + 2 * t);
        acc[j][0] = __uint_as_float(w0 << 16);
        acc[j][1] = __uint_as_float(w0 & 0xffff0000u);
        acc[j][2] = __uint_as_float(w8 << 16);
        acc[j][3] = __uint_as_float(w8 & 0xffff0000u);
      }
    }
    // clip (flagging non-finite values first), then per row half rr min / max over the quad's 64 values of
    // the group
    bool bad = false;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float tau = tau_s[8 * (8 * G + j) + 2 * t + (e & 1)];
        bad |= nonfinite(acc[j][e]) && ((checked >> (g + 8 * (e >> 1))) & 1u);
        acc[j][e] = fminf(fmaxf(acc[j][e], -tau), tau);
      }
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag(status, OSCAR_STATUS_NONFINITE);
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      float mn = acc[0][2 * rr], mx = mn;
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 2 * rr; e < 2 * rr + 2; ++e) {
          mn = fminf(mn, acc[j][e]);
          mx = fmaxf(mx, acc[j][e]);
        }
#pragma unroll
      for (int s = 1; s < 4; s <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, s));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
      }
      float sq, zq;
      uint32_t meta;
      if (mc == nullptr) {                          // fp16 (scale, zero), or (range, zero) with a codebook
        const float diff = __fsub_rn(mx, mn);
        const float scale = cb != nullptr ? diff : __fdiv_rn(diff, 3.0f);
        if ((fp16_saturates(scale) || fp16_saturates(mn)) && t == 0 && ((checked >> (g + 8 * rr)) & 1u))
          flag(status, OSCAR_STATUS_SATURATED);
        const __half2 sz = __halves2half2(__float2half_rn(sat_fp16(scale)), __float2half_rn(sat_fp16(mn)));
        sq = __low2float(sz);
        zq = __high2float(sz);
        meta = *reinterpret_cast<const uint32_t*>(&sz);
      } else {                                      // compact (mn8, mx8)
        unsigned mn8, mx8;
        u8_quant_params(mn, mx, mc[4 * G], mc[4 * G + 1], mc[4 * G + 2], mn8, mx8, sq, zq);
        meta = mn8 | (mx8 << 8);
      }
      const int row = g + 8 * rr;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t pair = 0;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float c = 0.f;
          if (sq != 0.f) {
            const float t = __fdiv_rn(__fsub_rn(acc[j][2 * rr + e], zq), sq);
            c = cb != nullptr ? cb_code(t, cb) : fminf(fmaxf(rintf(t), 0.f), 3.f);
          }
          pair |= ((uint32_t)c) << (8 * e);
        }
        *reinterpret_cast<uint16_t*>(codes_s + row * kD + 8 * (8 * G + j) + 2 * t) = (uint16_t)pair;
      }
      if (t == 0) meta_s[row * 2 + G] = meta;
    }
  }
}

// smem layout of one CTA (bytes): rotation fragments | tau | per warp: 2 staged tiles, codes, metadata
constexpr int kFragBytes = kRFragWords * 4;                               // 64 KB
constexpr int kTauBytes = kD * 4 + 32;           // tau, then the compact format's 8 grid constants
constexpr int kXTileBytes = kTileRows * kXStride * 2;                     // 4,352
constexpr int kWarpBytes = 2 * kXTileBytes + kTileRows * kD + kTileRows * 2 * 4;
constexpr int kPrefillMmaSmem = kFragBytes + kTauBytes + kPrefillWarps * kWarpBytes + 16;

__global__ void __launch_bounds__(kPrefillWarps * 32, 2)
    k_prefill_mma(LayerView lv, const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                  const int* __restrict__ cu_seqlens, int B, int total, const int* __restrict__ hist_pt,
                  int max_hist_pages, const int* __restrict__ bf16_pt) {
  TimelineSpan timeline_span(lv, kTlPrefill);
  extern __shared__ __align__(128) uint8_t smem[];
  uint32_t* frag_s = reinterpret_cast<uint32_t*>(smem);
  float* tau_s = reinterpret_cast<float*>(smem + kFragBytes);
  uint8_t* wbase = smem + kFragBytes + kTauBytes;
  const uint32_t bar = smem_addr(wbase + kPrefillWarps * kWarpBytes);
  __shared__ int landed;
  const int h = blockIdx.y, kind = blockIdx.z;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const bool rotate = (kind == OSCAR_KIND_K) || lv.v_explicit;
  const float* prm = lv.params + (size_t)h * kParamFloats;
  if (tid == 0) {
    landed = 1;
    if (rotate) {
      mbar_init(bar);
      bulk_load_hint(smem_addr(frag_s), prm + (kind == OSCAR_KIND_K ? kRKFragOff : kRVFragOff), kFragBytes, bar,
                     l2_evict_last());
    }
  }
  for (int i = tid; i < kD; i += blockDim.x) tau_s[i] = prm[(kind == OSCAR_KIND_K ? kTauKOff : kTauVOff) + i];
  if (tid < 8) tau_s[kD + tid] = prm[(lv.meta_cb ? kCbOff : kMetaCOff) + kind * 8 + tid];   // format constants
  const float* mc = lv.meta_u8 ? tau_s + kD : nullptr;
  const float* cbc = lv.meta_cb ? tau_s + kD : nullptr;
  __syncthreads();
  if (rotate && !__syncthreads_and(mbar_wait(bar, 0))) {
    if (tid == 0) flag(lv.status, OSCAR_STATUS_TIMEOUT);
    mbar_wait(bar, 0);                               // one more bounded wait for the copy in flight
    return;
  }
  const __nv_bfloat16* src_all = (kind == OSCAR_KIND_K) ? k : v;
  uint8_t* mine = wbase + w * kWarpBytes;
  uint8_t* codes_s = mine + 2 * kXTileBytes;
  uint32_t* meta_s = reinterpret_cast<uint32_t*>(codes_s + kTileRows * kD);
  const int tok0 = blockIdx.x * kPrefillTok, tok1 = min(tok0 + kPrefillTok, total);
  const int step = kPrefillWarps * kTileRows;
  int base = tok0 + w * kTileRows;
  auto xbuf = [&](int i) { return reinterpret_cast<__nv_bfloat16*>(mine + (i & 1) * kXTileBytes); };
  if (base < tok1) stage_tile(xbuf(0), src_all, base, tok1, h, lv.hkv);
  cp_async_commit();
  for (int it = 0; base < tok1; ++it, base += step) {
    // the next tile's rows are copied while this one is processed
    if (base + step < tok1) stage_tile(xbuf(it + 1), src_all, base + step, tok1, h, lv.hkv);
    cp_async_commit();
    const RowDest dst = lane < kTileRows ? classify(lv, base + lane, tok1, cu_seqlens, B, hist_pt, max_hist_pages,
                                                    bf16_pt)
                                         : RowDest{-1, 0, 0};
    cp_async_wait<1>();
    __syncwarp();
    const __nv_bfloat16* xs = xbuf(it);
    const uint32_t bf_rows = __ballot_sync(0xffffffffu, dst.where == 1);
    const uint32_t hist_rows = __ballot_sync(0xffffffffu, dst.where == 0);
    // sink / recent rows: bf16 copies
    for (uint32_t m = bf_rows; m != 0; m &= m - 1) {
      const int r = __ffs(m) - 1;
      const int page = __shfl_sync(0xffffffffu, dst.page, r), row = __shfl_sync(0xffffffffu, dst.row, r);
      __nv_bfloat16* out = bf16_row(lv, page, h, kind, row);
      const uint2 x = reinterpret_cast<const uint2*>(xs + r * kXStride)[lane];
      if (__any_sync(0xffffffffu, bf16x2_nonfinite(x.x) || bf16x2_nonfinite(x.y)) && lane == 0)
        flag(lv.status, OSCAR_STATUS_NONFINITE);
      reinterpret_cast<uint2*>(out)[lane] = x;
    }
    if (hist_rows != 0) {
      quantize_tile(frag_s, rotate, xs, tau_s, mc, cbc, codes_s, meta_s, lv.status, hist_rows);
      __syncwarp();
      if (kind == OSCAR_KIND_K) {
        // packed codes: 16 rows x 8 words of 16 codes; word idx = lane + 32 j
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int idx = lane + 32 * j, r = idx >> 3, wd = idx & 7;
          const int page = __shfl_sync(0xffffffffu, dst.page, r), row = __shfl_sync(0xffffffffu, dst.row, r);
          if (!((hist_rows >> r) & 1u)) continue;
          const uint32_t word = pack16(*reinterpret_cast<const uint4*>(codes_s + r * kD + 16 * wd));
          *reinterpret_cast<uint32_t*>(int2_block_w(lv, page, h) + kKCodesOff + row * (kD / 4) + 4 * wd) = word;
        }
      } else {
        // channel-major V: lane takes channels lane + 32 j; the tile's rows of one page are gathered per
        // 32-bit word of each channel (4 words a channel) and each word is updated by two atomics on its own
        // fields (a word may also hold rows of a neighbouring tile, written by another warp)
        uint8_t* cur = nullptr;
        unsigned msk[4][4], val[4][4];
        auto flush = [&]() {
          if (cur == nullptr) return;
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (msk[j][q] != 0u) {
                unsigned* wp = reinterpret_cast<unsigned*>(cur + v_chan_off(lane + 32 * j) + 4 * q);
                atomicAnd(wp, ~msk[j][q]);
                atomicOr(wp, val[j][q]);
              }
        };
        for (int r = 0; r < kTileRows; ++r) {
          if (!((hist_rows >> r) & 1u)) continue;  // warp-uniform
          const int page = __shfl_sync(0xffffffffu, dst.page, r), row = __shfl_sync(0xffffffffu, dst.row, r);
          uint8_t* blk = int2_block_w(lv, page, h);
          if (blk != cur) {
            flush();
            cur = blk;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
              for (int q = 0; q < 4; ++q) msk[j][q] = val[j][q] = 0u;
          }
          const int sh = v_bit(row), q0 = v_word(row);
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (q == q0) {
                msk[j][q] |= 3u << sh;
                val[j][q] |= (unsigned)codes_s[r * kD + lane + 32 * j] << sh;
              }
        }
        flush();
      }
      {
        const int r = lane >> 1, G = lane & 1;
        const int page = __shfl_sync(0xffffffffu, dst.page, r), row = __shfl_sync(0xffffffffu, dst.row, r);
        if ((hist_rows >> r) & 1u) {
          uint8_t* blk = int2_block_w(lv, page, h);
          if (mc == nullptr) {
            const int off = (kind == OSCAR_KIND_K ? kKMetaOff : kVMetaOff) + row * (kNG * 4) + G * 4;
            *reinterpret_cast<uint32_t*>(blk + off) = meta_s[r * 2 + G];
          } else {
            const int off = (kind == OSCAR_KIND_K ? kKMetaOff : kVMetaOffU8) + row * (kNG * 2) + G * 2;
            *reinterpret_cast<uint16_t*>(blk + off) = (uint16_t)meta_s[r * 2 + G];
          }
        }
      }
    }
    __syncwarp();                                   // this tile's buffers are free before the copy into them
  }
  cp_async_wait<0>();
}

}  // namespace

int launch_prefill(const LayerView& lv, int B, const void* k, const void* v, const int* cu_seqlens, int total,
                   const int* hist_pt, int max_hist_pages, const int* bf16_pt, cudaStream_t st) {
  if (total == 0 || B == 0) return OSCAR_OK;
  dim3 grid((total + kPrefillTok - 1) / kPrefillTok, lv.hkv, 2);
  k_prefill_mma<<<grid, kPrefillWarps * 32, kPrefillMmaSmem, st>>>(
      lv, static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), cu_seqlens, B, total, hist_pt,
      max_hist_pages, bf16_pt);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int configure_prefill_kernel() {
  return cudaFuncSetAttribute(k_prefill_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrefillMmaSmem) ==
                 cudaSuccess
             ? OSCAR_OK
             : OSCAR_ERR_CUDA;
}

}  // namespace oscar
