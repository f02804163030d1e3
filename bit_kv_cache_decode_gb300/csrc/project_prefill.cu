// Fused projection and write path on the 5th-generation tensor cores (sm_103a):
// K = x W_k^T and V = x W_v^T of the prompt's hidden states go straight into the
// pool, without a round trip of bf16 K and V through memory (MarkTechPost article
// "Together AI 开源 OSCAR…", section "服务系统：混合精度缓存布局": the write path
// runs fused; the same article: rotation, clipping, per-token asymmetric INT2,
// packed codes; news article "超越 TurboQuant…OSCAR…", section "OSCAR 的设计思路":
// prompt tokens land in the sink, the history and the recent window).
//
// k_project_prefill: one persistent CTA per SM; work items (tile, kind, head
// pair), items of a tile adjacent so that the CTAs working at one time share
// their x tiles in L2. A request's tokens form tiles of at most 128 rows of one
// role: its sink rows, its history rows from each page-pair boundary, its
// recent rows. Per item:
//  - warp 0 streams 64-wide slices of x (128 rows) and of W (256 rows: the two
//    heads) through a 4-stage ring by tensor-map copies (128-byte swizzle);
//  - warp 1 issues the GEMM: M = 128 rows, N = 256 channels, K = 16 per
//    instruction, float32 accumulation in TMEM columns 0-255;
//  - warps 2-9, the epilogue team, then take each head in turn: its 128
//    columns rounded to bf16 (to nearest even: the model's K and V); sink and
//    recent rows go to their BF16 page rows; history rows go to shared memory
//    as the A operand of Y = K R (R as three bf16 parts, or the identity for
//    V in V-absorbed mode; TMEM columns 256-383), then are quantised and
//    stored as the bulk prefill does. The pipeline's stages hold R and the A
//    operand meanwhile, so the next item's loads wait for the epilogue.
#include <algorithm>
#include <cuda.h>

#include "quant_tile.cuh"
#include "timeline.cuh"

namespace oscar {
namespace {

using namespace qtile;

constexpr int kPStages = 4;
constexpr int kXBox = kRows * 128;                     // 16 KB: 128 rows x 64 bf16
constexpr int kWBox = 2 * kD * 128;                    // 32 KB: 256 rows x 64 bf16
constexpr int kPStageBytes = kXBox + kWBox;            // 48 KB
constexpr int kOffR = 0;                               // epilogue: R image (96 KB) in stages 0-1
constexpr int kOffRotA = kRImgBytes;                   // epilogue: the rotation's A operand (32 KB)
constexpr int kOffCs = kOffRotA + 2 * kBoxBytes;       // epilogue: the transposing buffer
constexpr int kOffBar = kPStages * kPStageBytes;       // 196,608
// barriers: full[4], empty[4], gemm_done, r_full, rot_done, item_free, fin (GEMM), fin (rotations); then the
// TMEM address
constexpr int kBFull = 0, kBEmpty = kPStages, kBGemm = 2 * kPStages, kBRFull = kBGemm + 1, kBRot = kBGemm + 2,
              kBItemFree = kBGemm + 3, kBFin = kBGemm + 4, kBFinRot = kBGemm + 5, kNumPBars = kBFinRot + 1;
constexpr int kOffTiles = kOffBar + 128;               // int tile prefix over the requests [B + 1]
constexpr int kMaxProjBatch = 4096;
constexpr int kProjSmem = kOffTiles + 4 * (kMaxProjBatch + 1) + 1024;
constexpr int kProjThreads = 320;                      // loader, MMA, the 8-warp epilogue team
constexpr int kEpiBar = 1;                             // the team's named barrier
constexpr uint32_t kIdescGemm = idesc_f16(128, 256) | (1u << 7) | (1u << 10);   // bf16, M 128, N 256
constexpr uint32_t kColRot = 256;

static_assert(kOffCs + kCsBytes <= kOffBar, "epilogue buffers fit in the ring");
static_assert(kNumPBars * 8 + 4 <= kOffTiles - kOffBar, "barriers and the TMEM address");
static_assert(kProjSmem <= 232448, "shared memory");

enum Role : int { kSink = 0, kHist = 1, kRecent = 2 };

// request r's tiles: its sink rows (one tile), history tiles of 128 rows, recent tiles of 128 rows
__device__ __forceinline__ void req_split(const LayerView& lv, const int* cu, int r, int& ns, int& nh, int& nr) {
  const int L = cu[r + 1] - cu[r];
  ns = min(L, lv.sink);
  nh = max(0, L - lv.sink - lv.recent);
  nr = L - ns - nh;
}
__device__ __forceinline__ int req_ntiles(const LayerView& lv, const int* cu, int r) {
  int ns, nh, nr;
  req_split(lv, cu, r, ns, nh, nr);
  return (ns > 0 ? 1 : 0) + (nh + kRows - 1) / kRows + (nr + kRows - 1) / kRows;
}

struct Tile {
  int r, role, tok0, rows, h0;    // request, role, first token (in the request), rows, first history row
};
// tile t of the batch (prefix[r] = tiles before request r, in shared memory)
__device__ Tile tile_of(const LayerView& lv, const int* cu, const int* prefix, int B, int t) {
  int lo = 0, hi = B - 1;                         // the last r with prefix[r] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  Tile x;
  x.r = lo;
  int j = t - prefix[lo], ns, nh, nr;
  req_split(lv, cu, lo, ns, nh, nr);
  x.h0 = 0;
  if (ns > 0 && j == 0) {
    x.role = kSink;
    x.tok0 = 0;
    x.rows = ns;
    return x;
  }
  j -= ns > 0 ? 1 : 0;
  const int th = (nh + kRows - 1) / kRows;
  if (j < th) {
    x.role = kHist;
    x.h0 = kRows * j;
    x.tok0 = lv.sink + x.h0;
    x.rows = min(kRows, nh - x.h0);
    return x;
  }
  j -= th;
  x.role = kRecent;
  x.tok0 = ns + nh + kRows * j;
  x.rows = min(kRows, nr - kRows * j);
  return x;
}

template <int FMT>
__global__ void __launch_bounds__(kProjThreads, 1)
    k_project_prefill(LayerView lv, const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_wk,
                      const __grid_constant__ CUtensorMap map_wv, const int* __restrict__ cu_seqlens, int B,
                      int d_model, const int* __restrict__ hist_pt, int max_hist_pages,
                      const int* __restrict__ bf16_pt) {
  TimelineSpan timeline_span(lv, kTlPrefill);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sb = smem_addr(smem);
  auto bar = [&](int i) { return sb + (uint32_t)kOffBar + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + kNumPBars * 8);
  int* prefix = reinterpret_cast<int*>(smem + kOffTiles);

  if (tid == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init_n(bar(kBFull + s), 1);
      mbar_init_n(bar(kBEmpty + s), 1);
    }
    mbar_init_n(bar(kBGemm), 1);
    mbar_init_n(bar(kBRFull), 1);
    mbar_init_n(bar(kBRot), 1);
    mbar_init_n(bar(kBItemFree), 1);
    mbar_init_n(bar(kBFin), 1);
    mbar_init_n(bar(kBFinRot), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (warp == 2) {                                 // the tile prefix over the requests
    int carry = 0;
    for (int r0 = 0; r0 < B; r0 += 32) {
      const int nt = r0 + lane < B ? req_ntiles(lv, cu_seqlens, r0 + lane) : 0;
      int incl = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
      }
      if (r0 + lane < B) prefix[r0 + lane] = carry + incl - nt;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) prefix[B] = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int T = prefix[B];
  const int pairs = lv.hkv / 2, per_tile = 2 * pairs;
  const long long N = (long long)T * per_tile;
  const int cnt = N > blockIdx.x ? (int)((N - 1 - blockIdx.x) / gridDim.x) + 1 : 0;
  const int nk = d_model / 64;
  bool ok = true;

  if (cnt > 0 && warp == 0) {
    // ---- loader: for each item, the x and W slices (after the previous item's epilogue is done) ----
    const uint64_t pol_x = l2_evict_normal(), pol_w = l2_evict_last();   // x tiles: read by a tile's items
    int issued = 0;
    for (int i = 0; i < cnt && ok; ++i) {
      const long long n = blockIdx.x + (long long)i * gridDim.x;
      const int t = (int)(n / per_tile), kp = (int)(n % per_tile), kind = kp / pairs, hp = kp % pairs;
      const Tile tl = tile_of(lv, cu_seqlens, prefix, B, t);
      const int row0 = cu_seqlens[tl.r] + tl.tok0;
      const CUtensorMap* wmap = kind == OSCAR_KIND_K ? &map_wk : &map_wv;
      if (i > 0) {
        bool good = lane == 0 ? mbar_wait(bar(kBItemFree), (i - 1) & 1) : true;
        if (!__shfl_sync(0xffffffffu, good, 0)) {
          ok = false;
          break;
        }
      }
      for (int ks = 0; ks < nk; ++ks, ++issued) {
        const int s = issued % kPStages;
        bool good = true;
        if (lane == 0) {
          good = mbar_wait(bar(kBEmpty + s), ((issued / kPStages) & 1) ^ 1);
          if (good) {
            const uint32_t dst = sb + s * kPStageBytes;
            mbar_expect_tx(bar(kBFull + s), kPStageBytes);
            tma_load_2d(dst, &map_x, 64 * ks, row0, bar(kBFull + s), pol_x);
            tma_load_2d(dst + kXBox, wmap, 64 * ks, 2 * kD * hp, bar(kBFull + s), pol_w);
          }
        }
        if (!__shfl_sync(0xffffffffu, good, 0)) {
          ok = false;
          break;
        }
      }
    }
    // every copy this warp issued lands before the CTA may exit
    if (lane == 0)
      for (int k = max(0, issued - kPStages); k < issued; ++k)
        if (!mbar_wait(bar(kBFull + k % kPStages), (k / kPStages) & 1)) ok = false;
  } else if (cnt > 0 && warp == 1) {
    // ---- GEMM issue: D[0, 256) = x W^T over d_model ----
    int used = 0;
    for (int i = 0; i < cnt && ok; ++i) {
      for (int ks = 0; ks < nk; ++ks, ++used) {
        const int s = used % kPStages;
        bool good = true;
        if (lane == 0) good = mbar_wait(bar(kBFull + s), (used / kPStages) & 1);
        if (!__shfl_sync(0xffffffffu, good, 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = sb + s * kPStageBytes, b0 = a0 + kXBox;
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            umma(tmem, desc_sw128(a0 + 32 * k4), desc_sw128(b0 + 32 * k4), kIdescGemm, (ks | k4) != 0);
          umma_commit(bar(kBEmpty + s));         // the stage is free once these MMAs complete
          if (ks == nk - 1) umma_commit(bar(kBGemm));
        }
        __syncwarp();
      }
    }
    if (lane == 0) {                             // every MMA has completed before TMEM is released
      umma_commit(bar(kBFin));
      if (!mbar_wait(bar(kBFin), 0)) ok = false;
    }
  } else if (cnt > 0) {
    // ---- epilogue team: warp (lane quarter q, half / group G), row = 32 q + lane ----
    const int e = warp - 2, q = warp & 3, G = e >> 2;
    const int row = 32 * q + lane, u = e * 32 + lane;
    const uint32_t tl_lane = tmem + ((uint32_t)(32 * q) << 16);
    uint8_t* rota = smem + kOffRotA;
    uint8_t* cs = smem + kOffCs;
    int nrot = 0;                                  // rotations so far (phases of r_full and rot_done)
    const int bpr = (lv.sink + lv.recent) / kP;
    for (int i = 0; i < cnt; ++i) {
      const long long n = blockIdx.x + (long long)i * gridDim.x;
      const int t = (int)(n / per_tile), kp = (int)(n % per_tile), kind = kp / pairs, hp = kp % pairs;
      const Tile tl = tile_of(lv, cu_seqlens, prefix, B, t);
      if (!named_and(kEpiBar, kTeamThreads, mbar_wait(bar(kBGemm), i & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      bool good = true;
      for (int hh = 0; hh < 2 && good; ++hh) {
        const int h = 2 * hp + hh;
        const bool rotate = kind == OSCAR_KIND_K || lv.v_explicit;
        if (tl.role == kHist) {
          // the head's B operand (the GEMM's stages and the previous rotation are done with this memory)
          if (rotate) {
            if (u == 0) {
              const uint8_t* img = reinterpret_cast<const uint8_t*>(
                  lv.params + (size_t)h * kParamFloats + (kind == OSCAR_KIND_K ? kRKImgOff : kRVImgOff));
              mbar_expect_tx(bar(kBRFull), kRImgBytes);
              for (int c = 0; c < 3; ++c) bulk_copy(sb + kOffR + c * 32768, img + c * 32768, 32768, bar(kBRFull));
            }
          } else {                                 // the identity: V stored as it comes
            uint4* z = reinterpret_cast<uint4*>(smem + kOffR);
            for (int x = u; x < 32768 / 16; x += kTeamThreads) z[x] = make_uint4(0u, 0u, 0u, 0u);
            named_sync(kEpiBar, kTeamThreads);
            if (u < kD) *reinterpret_cast<uint16_t*>(smem + kOffR + sw128_offset(u, u)) = 0x3F80;   // bf16 1.0
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            named_sync(kEpiBar, kTeamThreads);
            if (u == 0) mbar_arrive(bar(kBRFull));
          }
        }
        // the head's 64 channels of this warp, rounded to bf16
        __syncwarp();
        uint32_t pk[32];
        {
          float a[32], b[32];
          tmem_ld32x2(tl_lane + 128u * hh + 64u * G, tl_lane + 128u * hh + 64u * G + 32u, a, b);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(a[2 * j], a[2 * j + 1]);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(b[2 * j], b[2 * j + 1]);
            pk[j] = *reinterpret_cast<const uint32_t*>(&lo);
            pk[16 + j] = *reinterpret_cast<const uint32_t*>(&hi);
          }
        }
        const bool row_ok = row < tl.rows;
        bool nf = false;
#pragma unroll
        for (int j = 0; j < 32; ++j) nf |= bf16x2_nonfinite(pk[j]);
        if (tl.role != kHist) {
          // sink / recent rows: the BF16 page row (channels 64 G ..)
          if (__any_sync(0xffffffffu, row_ok && nf) && lane == 0) flag(lv.status, OSCAR_STATUS_NONFINITE);
          if (row_ok) {
            const int pos = tl.tok0 + row;
            int page, prow;
            if (tl.role == kSink) {
              page = bf16_pt[(size_t)tl.r * bpr + pos / kP];
              prow = pos % kP;
            } else {
              const int slot = (pos - lv.sink) % lv.recent;
              page = bf16_pt[(size_t)tl.r * bpr + lv.sink / kP + slot / kP];
              prow = slot % kP;
            }
            if (page < 0 || page >= lv.n_bf16) {
              flag(lv.status, OSCAR_STATUS_BAD_PAGE);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(bf16_row(lv, page, h, kind, prow) + 64 * G);
#pragma unroll
              for (int c8 = 0; c8 < 8; ++c8) dst[c8] = make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
            }
          }
          continue;
        }
        // history rows: the rotation's A operand (row `row`, channel half G, 128-byte swizzle)
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)
          *reinterpret_cast<uint4*>(rota + G * kBoxBytes + row * 128 + ((c8 ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        named_sync(kEpiBar, kTeamThreads);
        if (u == 0) {
          if (mbar_wait(bar(kBRFull), nrot & 1)) {
            tc_fence_after();
            const uint32_t a0 = sb + kOffRotA, b0 = sb + kOffR;
            const int parts = rotate ? 3 : 1;
            for (int p = 0; p < parts; ++p)
#pragma unroll
              for (int kh = 0; kh < 2; ++kh)
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4)
                  umma(tmem + kColRot, desc_sw128(a0 + kh * kBoxBytes + 32 * k4),
                       desc_sw128(b0 + p * 32768 + kh * kBoxBytes + 32 * k4), kIdescBf16, (p | kh | k4) != 0);
            umma_commit(bar(kBRot));
          }
        }
        good = named_and(kEpiBar, kTeamThreads, mbar_wait(bar(kBRot), nrot & 1));
        ++nrot;
        if (!good) break;
        tc_fence_after();
        uint32_t wd[4], meta;
        bool nfq, sat;
        quantise_group<FMT>(tl_lane + kColRot + 64u * G, lv.params + (size_t)h * kParamFloats, kind, G, wd, meta,
                            nfq, sat);
        store_history_row<FMT>(lv, hist_pt, max_hist_pages, tl.r, h, kind, tl.h0, tl.rows, row, G, u, wd, meta,
                               nfq || nf, sat, cs, kEpiBar);
        // the rotation's columns, A operand, B operand and transposing buffer are free for the next head
        tc_fence_before();
        named_sync(kEpiBar, kTeamThreads);
      }
      if (!good) {
        ok = false;
        break;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the ring is rewritten by copies next
      tc_fence_before();
      named_sync(kEpiBar, kTeamThreads);
      if (u == 0) mbar_arrive(bar(kBItemFree));  // the accumulator and the ring are free for the next item
    }
    if (u == 0 && nrot > 0) {                    // the rotations this thread issued have completed
      umma_commit(bar(kBFinRot));
      if (!mbar_wait(bar(kBFinRot), 0)) ok = false;
    }
  }
  if (!ok && lane == 0) flag(lv.status, OSCAR_STATUS_TIMEOUT);
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

// a row-major bf16 matrix [rows][cols] as a 2-D tensor; boxes of 64 columns x box_rows rows land
// 128-byte swizzled; rows past the end read as zero
bool matrix_map(CUtensorMap* map, const void* base, long long rows, int cols, int box_rows) {
  EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_project_prefill(const LayerView& lv, int B, const void* x, int d_model, const void* w_k, const void* w_v,
                           const int* cu_seqlens, int total, const int* hist_pt, int max_hist_pages,
                           const int* bf16_pt, cudaStream_t st) {
  if (total == 0 || B == 0) return OSCAR_OK;
  if (lv.hkv % 2 != 0 || d_model % 64 != 0 || d_model <= 0 || B > kMaxProjBatch) return OSCAR_ERR_UNSUPPORTED;
  CUtensorMap mx, mk, mv;
  if (!matrix_map(&mx, x, total, d_model, kRows) || !matrix_map(&mk, w_k, (long long)lv.hkv * kD, d_model, 2 * kD) ||
      !matrix_map(&mv, w_v, (long long)lv.hkv * kD, d_model, 2 * kD))
    return OSCAR_ERR_CUDA;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // at most one tile per 64 tokens plus three per request; one CTA per SM
  const long long items_max = (long long)lv.hkv * ((long long)total / kP + 3LL * B);
  const int grid = (int)std::max(1LL, std::min((long long)sms, items_max));
  if (lv.meta_u8)
    k_project_prefill<kFmtU8><<<grid, kProjThreads, kProjSmem, st>>>(lv, mx, mk, mv, cu_seqlens, B, d_model, hist_pt,
                                                                       max_hist_pages, bf16_pt);
  else if (lv.meta_cb)
    k_project_prefill<kFmtCB><<<grid, kProjThreads, kProjSmem, st>>>(lv, mx, mk, mv, cu_seqlens, B, d_model, hist_pt,
                                                                       max_hist_pages, bf16_pt);
  else
    k_project_prefill<kFmtF16><<<grid, kProjThreads, kProjSmem, st>>>(lv, mx, mk, mv, cu_seqlens, B, d_model, hist_pt,
                                                                        max_hist_pages, bf16_pt);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int configure_project_prefill_kernel() {
  const bool ok =
      cudaFuncSetAttribute(k_project_prefill<kFmtF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kProjSmem) ==
          cudaSuccess &&
      cudaFuncSetAttribute(k_project_prefill<kFmtU8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kProjSmem) ==
          cudaSuccess &&
      cudaFuncSetAttribute(k_project_prefill<kFmtCB>, cudaFuncAttributeMaxDynamicSharedMemorySize, kProjSmem) ==
          cudaSuccess;
  return ok ? OSCAR_OK : OSCAR_ERR_CUDA;
}

}  // namespace oscar
