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
//  * k_prefill_hist quantises the history. grid (nx, kv head, K / V), 128
//    threads, persistent over the history tiles of all requests: a tile is 128
//    history rows of one request starting at a page pair boundary, so a tile
//    owns its pages' code and metadata bytes outright. Per tile:
//    - the rows arrive by bulk copies into shared memory (row = thread);
//    - rotated kinds (K always, V in explicit-V mode): the thread converts its
//      row to fp16 (exact for bf16 values of normal fp16 range) and stores it in
//      tensor memory, the A operand of Y = X R; R = U H P_br (composed on the
//      host) sits in shared memory as fp16 high and low parts in the no-swizzle
//      K-major layout, and one thread issues 16 tcgen05.mma (M = 128 rows, N =
//      128 rotated channels, K = 16): Y = X R_hi + X R_lo accumulates in tensor
//      memory;
//    - the thread reads its row of Y and quantises it: clip to +-tau, group
//      min / max, the format's scale and zero, codes, each step the same float32
//      operation as in the single-row quantiser;
//    - K codes and all metadata go straight to the page rows; V codes, which
//      are channel-major, are gathered in shared memory and written one 16-byte
//      channel slot per thread.
#include <algorithm>

#include "kernels.cuh"
#include "rotate.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"
#include "timeline.cuh"

namespace oscar {
namespace {

constexpr int kTile = 2 * kP;                       // history rows per tile
constexpr int kXRow = kD * 2 + 16;                  // staged row: 272 bytes, conflict-free 16-byte loads
constexpr int kRPart = kD * kD * 2;                 // 32 KB: one fp16 part of R, K-major canonical
constexpr int kRSbo = (kD / 8) * 128;               // 2,048: 8-row blocks of the canonical layout
constexpr int kOffR = 0;                            // R_hi, R_lo
constexpr int kOffX = 2 * kRPart;                   // staged rows, then (after the A operand is built) the V codes
constexpr int kOffTau = kOffX + kTile * kXRow;      // tau[128], then the format constants [8]
constexpr int kOffBar = kOffTau + (kD + 8) * 4;
constexpr int kPrefSmem = kOffBar + 16 + 16 + 1024;
constexpr uint32_t kPrefCols = 256, kColA = 0, kColY = 128;
constexpr uint32_t kIdescN128 = idesc_f16(128, 128);

__device__ __forceinline__ int canon_r(int n, int k) {
  return (n >> 3) * kRSbo + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2;
}
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// tiles of request r: ceil(history rows / 128); the whole batch's prefix sums
__device__ __forceinline__ int hist_rows(const LayerView& lv, const int* cu, int r) {
  return max(0, cu[r + 1] - cu[r] - lv.sink - lv.recent);
}

__global__ void __launch_bounds__(128, 2) k_prefill_hist(LayerView lv, const __nv_bfloat16* __restrict__ k,
                                                         const __nv_bfloat16* __restrict__ v,
                                                         const int* __restrict__ cu_seqlens, int B,
                                                         const int* __restrict__ hist_pt, int max_hist_pages) {
  TimelineSpan timeline_span(lv, kTlPrefill);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int h = blockIdx.y, kind = blockIdx.z;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const bool rotate = kind == OSCAR_KIND_K || lv.v_explicit;
  const float* prm = lv.params + (size_t)h * kParamFloats;
  float* tau_s = reinterpret_cast<float*>(smem + kOffTau);
  const uint32_t bar = smem_addr(smem + kOffBar), bar_mma = bar + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 16);
  const __nv_bfloat16* src = kind == OSCAR_KIND_K ? k : v;
  const float* mc = lv.meta_u8 ? tau_s + kD : nullptr;
  const float* cbc = lv.meta_cb ? tau_s + kD : nullptr;

  // ---- set-up: R's two fp16 parts in the canonical layout, tau, the format constants, TMEM ----
  if (rotate) {
    // the fragment words (mma.m16n8k16 B order: k-block kb, n-tile nt, lane (g, t), {hi b0, hi b1, lo b0, lo b1})
    // become element pairs (n = 8 nt + g, k = 16 kb + 2t (+ 8), + 1) of the canonical layout
    const uint32_t* frag = reinterpret_cast<const uint32_t*>(prm + (kind == OSCAR_KIND_K ? kRKFragOff : kRVFragOff));
    for (int wi = tid; wi < kRFragWords; wi += 128) {
      const int e = wi & 3, ln = (wi >> 2) & 31, nt = (wi >> 7) & 15, kb = wi >> 11;
      const int n = 8 * nt + (ln >> 2), kk = 16 * kb + 2 * (ln & 3) + 8 * (e & 1);
      *reinterpret_cast<uint32_t*>(smem + kOffR + (e >> 1) * kRPart + canon_r(n, kk)) = __ldg(frag + wi);
    }
  }
  for (int i = tid; i < kD; i += 128) tau_s[i] = prm[(kind == OSCAR_KIND_K ? kTauKOff : kTauVOff) + i];
  if (tid < 8) tau_s[kD + tid] = prm[(lv.meta_cb ? kCbOff : kMetaCOff) + kind * 8 + tid];
  if (tid == 0) {
    mbar_init_n(bar, 1);
    mbar_init_n(bar_mma, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (w == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kPrefCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");     // the MMAs read R
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tl = tmem + ((uint32_t)(32 * w) << 16);

  // ---- the tiles: t = blockIdx.x, + gridDim.x, ... over the batch's history tiles ----
  int total = 0;
  for (int r = 0; r < B; ++r) total += (hist_rows(lv, cu_seqlens, r) + kTile - 1) / kTile;
  uint32_t phase = 0;
  bool ok = true;
  for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
    int r = 0, j = t;                              // request r, its tile j
    for (;;) {
      const int n = (hist_rows(lv, cu_seqlens, r) + kTile - 1) / kTile;
      if (j < n) break;
      j -= n;
      ++r;
    }
    const int hn = min(kTile, hist_rows(lv, cu_seqlens, r) - kTile * j);   // rows of this tile
    const int h0 = kTile * j;                      // first history row
    const bool row_ok = tid < hn;
    // this thread's destination page and row; a bad page id skips the row (and is flagged)
    const int hp = (h0 + tid) / kP;
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
    // ---- the rows into shared memory ----
    uint8_t* xs = smem + kOffX;
    if (tid == 0) mbar_expect_tx(bar, (uint32_t)(hn * kD * 2));
    __syncthreads();                               // the bytes are announced before any copy can complete
    if (row_ok) {
      const size_t tok = (size_t)cu_seqlens[r] + lv.sink + h0 + tid;
      bulk_copy(smem_addr(xs + tid * kXRow), src + (tok * lv.hkv + h) * kD, kD * 2, bar);
    }
    ok = __syncthreads_and(mbar_wait(bar, phase));
    phase ^= 1u;
    if (!ok) {
      if (tid == 0) flag(lv.status, OSCAR_STATUS_TIMEOUT);
      break;
    }
    const uint4* xr = reinterpret_cast<const uint4*>(xs + tid * kXRow);
    float y[kD];
    if (rotate) {
      // A = the row as fp16 pairs (channels 2c, 2c + 1 in TMEM column c), then Y = X R_hi + X R_lo
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t a[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 x = row_ok ? xr[8 * half + q] : make_uint4(0u, 0u, 0u, 0u);
          a[4 * q] = bf16x2_to_f16x2(x.x);
          a[4 * q + 1] = bf16x2_to_f16x2(x.y);
          a[4 * q + 2] = bf16x2_to_f16x2(x.z);
          a[4 * q + 3] = bf16x2_to_f16x2(x.w);
        }
        tmem_st32u(tl + kColA + 32 * half, a);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncthreads();                             // every row's A is in; the staged rows are free
      if (tid == 0) {
        tc_fence_after();
        const uint32_t ra = smem_addr(smem + kOffR);
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int s = 0; s < 8; ++s)              // input channels 16 s .. 16 s + 15
            umma_ta(tmem + kColY, tmem + kColA + 8 * s, umma_desc(ra + part * kRPart + 2 * s * 128, 128, kRSbo),
                    kIdescN128, part > 0 || s > 0);
        umma_commit(bar_mma);
      }
      ok = __syncthreads_and(mbar_wait(bar_mma, (phase >> 1) & 1u));
      phase ^= 2u;
      if (!ok) {
        if (tid == 0) flag(lv.status, OSCAR_STATUS_TIMEOUT);
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float v32[32];
        tmem_ld32(tl + kColY + 32 * c4, v32);
#pragma unroll
        for (int i = 0; i < 32; ++i) y[32 * c4 + i] = v32[i];
      }
    } else {
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const uint4 x = row_ok ? xr[q] : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          y[8 * q + 2 * e] = __uint_as_float(wd[e] << 16);
          y[8 * q + 2 * e + 1] = __uint_as_float(wd[e] & 0xffff0000u);
        }
      }
      __syncthreads();                             // the staged rows are free
    }
    // ---- quantise this row: clip, group min / max, scale / zero, codes ----
    uint32_t packed[8];                            // 16 codes per word, channel 16 q + m at bits 2m
    uint32_t meta[2];
    bool bad = false;
#pragma unroll
    for (int G = 0; G < 2; ++G) {
      float mn = INFINITY, mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const int ch = 64 * G + i;
        bad |= nonfinite(y[ch]);
        const float tt = tau_s[ch];
        y[ch] = fminf(fmaxf(y[ch], -tt), tt);
        mn = fminf(mn, y[ch]);
        mx = fmaxf(mx, y[ch]);
      }
      float sq, zq;
      if (mc == nullptr) {                         // fp16 (scale, zero), or (range, zero) with a codebook
        const float diff = __fsub_rn(mx, mn);
        const float scale = cbc != nullptr ? diff : __fdiv_rn(diff, 3.0f);
        if ((fp16_saturates(scale) || fp16_saturates(mn)) && row_ok) flag(lv.status, OSCAR_STATUS_SATURATED);
        const __half2 sz = __halves2half2(__float2half_rn(sat_fp16(scale)), __float2half_rn(sat_fp16(mn)));
        sq = __low2float(sz);
        zq = __high2float(sz);
        meta[G] = *reinterpret_cast<const uint32_t*>(&sz);
      } else {                                     // compact (mn8, mx8)
        unsigned mn8, mx8;
        u8_quant_params(mn, mx, mc[4 * G], mc[4 * G + 1], mc[4 * G + 2], mn8, mx8, sq, zq);
        meta[G] = mn8 | (mx8 << 8);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t word = 0u;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const int ch = 64 * G + 16 * q + m;
          float c = 0.f;
          if (sq != 0.f) {
            const float tq = __fdiv_rn(__fsub_rn(y[ch], zq), sq);
            c = cbc != nullptr ? cb_code(tq, cbc) : fminf(fmaxf(rintf(tq), 0.f), 3.f);
          }
          word |= ((uint32_t)c) << (2 * m);
        }
        packed[4 * G + q] = word;
      }
    }
    if (bad && row_ok) flag(lv.status, OSCAR_STATUS_NONFINITE);
    // ---- K codes and every row's metadata straight to the page rows; V codes through shared memory ----
    uint8_t* blk = page >= 0 ? int2_block_w(lv, page, h) : nullptr;
    const int prow = (h0 + tid) % kP;
    if (blk != nullptr) {
      if (kind == OSCAR_KIND_K) {
        uint4* dst = reinterpret_cast<uint4*>(blk + kKCodesOff + prow * (kD / 4));
        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
      }
      if (mc == nullptr) {
        *reinterpret_cast<uint2*>(blk + (kind == OSCAR_KIND_K ? kKMetaOff : kVMetaOff) + prow * (kNG * 4)) =
            make_uint2(meta[0], meta[1]);
      } else {
        *reinterpret_cast<uint32_t*>(blk + (kind == OSCAR_KIND_K ? kKMetaOff : kVMetaOffU8) + prow * (kNG * 2)) =
            (meta[0] & 0xffffu) | (meta[1] << 16);
      }
    }
    if (kind == OSCAR_KIND_V) {
      // the rows' codes [128 rows][32 bytes] in shared memory (rows past the tile: zero), then thread c writes
      // channel c's 16-byte slot of each page of the tile
      uint8_t* cs = smem + kOffX;
      uint4* dst = reinterpret_cast<uint4*>(cs + tid * 32);
      dst[0] = row_ok ? make_uint4(packed[0], packed[1], packed[2], packed[3]) : make_uint4(0u, 0u, 0u, 0u);
      dst[1] = row_ok ? make_uint4(packed[4], packed[5], packed[6], packed[7]) : make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      const int c = tid;
      for (int pg = 0; pg < 2; ++pg) {
        if (pg * kP >= hn) break;
        const int pid = (h0 / kP + pg) < max_hist_pages ? hist_pt[(size_t)r * max_hist_pages + h0 / kP + pg] : -1;
        if (pid < 0 || pid >= lv.n_int2) continue;  // flagged by the rows above
        uint32_t wv[4] = {0u, 0u, 0u, 0u};
        // row t of the page: word (t >> 1) & 3, bit v_bit(t)
        for (int tr = 0; tr < kP; ++tr) {
          const int row = pg * kP + tr;
          const uint32_t code = (cs[row * 32 + (c >> 2)] >> (2 * (c & 3))) & 3u;
          wv[v_word(tr)] |= code << v_bit(tr);
        }
        *reinterpret_cast<uint4*>(int2_block_w(lv, pid, h) + v_chan_off(c)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
    }
    __syncthreads();                               // the staging buffer is free for the next tile
  }
  tc_fence_before();
  __syncthreads();
  if (w == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPrefCols) : "memory");
  }
}

// Sink and recent rows of request r, kv head h, one kind: bf16 copies, one warp per row.
__global__ void __launch_bounds__(128) k_prefill_bf16(LayerView lv, const __nv_bfloat16* __restrict__ k,
                                                      const __nv_bfloat16* __restrict__ v,
                                                      const int* __restrict__ cu_seqlens, const int* __restrict__ bf16_pt) {
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

int launch_prefill(const LayerView& lv, int B, const void* k, const void* v, const int* cu_seqlens, int total,
                   const int* hist_pt, int max_hist_pages, const int* bf16_pt, cudaStream_t st) {
  if (total == 0 || B == 0) return OSCAR_OK;
  const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(k);
  const __nv_bfloat16* vb = static_cast<const __nv_bfloat16*>(v);
  k_prefill_bf16<<<dim3(B, lv.hkv, 2), 128, 0, st>>>(lv, kb, vb, cu_seqlens, bf16_pt);
  // two CTAs per SM over the (kv head, kind) pairs, each walking its share of the batch's history tiles
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int tiles_max = total / kTile + B;
  const int nx = std::max(1, std::min(tiles_max, (2 * sms) / (2 * lv.hkv)));
  k_prefill_hist<<<dim3(nx, lv.hkv, 2), 128, kPrefSmem, st>>>(lv, kb, vb, cu_seqlens, B, hist_pt, max_hist_pages);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int configure_prefill_kernel() {
  return cudaFuncSetAttribute(k_prefill_hist, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrefSmem) == cudaSuccess
             ? OSCAR_OK
             : OSCAR_ERR_CUDA;
}

}  // namespace oscar
