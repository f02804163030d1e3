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

#include "quant_tile.cuh"
#include "timeline.cuh"

namespace oscar {
namespace {

using namespace qtile;

constexpr int kTile = kRows;                           // history rows per tile
// relative cost of a K and a V item (a tile of one kind and head), from the CTAs' end times on the
// 911,226-token Qwen3-32B-shaped batch: in V-absorbed mode a K item (24 MMAs) takes about 6 % longer
// than a V item (8 MMAs and the channel transpose); in explicit-V mode a V item (rotation and transpose)
// about 8 % longer than a K item
constexpr long long kCostK = 106, kCostV = 100, kCostRot = 100, kCostVRot = 108;
constexpr int kStages = 3;
constexpr int kStageBytes = 2 * kBoxBytes;             // 32 KB
constexpr int kYBufs = 4;                              // TMEM accumulators of 128 columns
constexpr int kTeams = 2;
constexpr int kThreads = 64 + kTeams * kTeamThreads;   // 576: loader, MMA, two epilogue teams
constexpr int kOffStage = 0;
constexpr int kOffB = kOffStage + kStages * kStageBytes;          // 98,304
constexpr int kOffCs = kOffB + kRImgBytes;                         // 196,608: [team][kCsBytes]
constexpr int kOffBar = kOffCs + kTeams * kCsBytes;               // 205,056
// barriers: full[3], empty[3], b_full, b_free, y_full[4], y_empty[4], fin; then the TMEM address
constexpr int kBarFull = 0, kBarEmpty = kStages, kBarBFull = 2 * kStages, kBarBFree = kBarBFull + 1,
              kBarYFull = kBarBFree + 1, kBarYEmpty = kBarYFull + kYBufs, kBarFin = kBarYEmpty + kYBufs,
              kNumBars = kBarFin + 1;
constexpr int kPrefSmem = kOffBar + kNumBars * 8 + 8 + 1024;       // + alignment slack
static_assert(kPrefSmem <= 232448, "shared memory");

// named barriers of the two epilogue teams: ids 1, 2
__device__ __forceinline__ bool team_and(int team, bool p) { return named_and(1 + team, kTeamThreads, p); }

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
  // CTA x takes the items of cost share [x W / grid, (x + 1) W / grid): the K items come first and cost
  // kCostK each, the V items kCostV (V-absorbed: no rotation; explicit V: the rotation and the channel
  // transpose), so that the CTAs of both kinds end together
  const long long nk = (long long)lv.hkv * T;
  const long long ck = lv.v_explicit ? kCostRot : kCostK, cv = lv.v_explicit ? kCostVRot : kCostV;
  const long long W = nk * (ck + cv);
  auto item_at = [&](long long cost) { return cost <= nk * ck ? cost / ck : nk + (cost - nk * ck) / cv; };
  const long long n0 = item_at(W * blockIdx.x / gridDim.x);
  const long long n1 = blockIdx.x + 1 == gridDim.x ? 2 * nk : item_at(W * (blockIdx.x + 1) / gridDim.x);
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
        const float* prm = lv.params + (size_t)h * kParamFloats;
        uint32_t wd[4], meta;
        bool nf, sat;
        quantise_group<FMT>(tmem + ((uint32_t)(32 * q) << 16) + 128u * b + 64u * G, prm, kind, G, wd, meta, nf,
                            sat);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarYEmpty + b));   // the accumulator is free for the MMA
        store_history_row<FMT>(lv, hist_pt, max_hist_pages, r, h, kind, h0, hn, row, G, u, wd, meta, nf, sat, cs,
                               1 + team);
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
  // the sink / recent copy runs beside the history kernel: with the largest shared-memory carveout an SM
  // running one of its CTAs can also take a history CTA (206 KB) instead of waiting for it to finish
  if (cudaFuncSetAttribute(k_prefill_bf16, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    return OSCAR_ERR_CUDA;
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
