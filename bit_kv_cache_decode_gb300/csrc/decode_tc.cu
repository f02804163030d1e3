// INT2 history decode on the 5th-generation tensor cores (sm_103a): tcgen05.mma
// with the unpacked codes as the A operand in tensor memory.
//
// News article "超越 TurboQuant…OSCAR…", section "OSCAR 的设计思路": the INT2
// kernel unpacks the 2-bit codes, restores scale/zero and accumulates in
// floating point; MarkTechPost article "Together AI 开源 OSCAR…", section "服务
// 系统：混合精度缓存布局": packed codes, per-token groups of 64 channels.
//
// Work: grid (split + 1, kv head, request), 256 threads. A history CTA takes the
// pages [p0, p1) of its split in tiles of two pages (128 tokens); the last CTA
// of each (request, kv head) attends its BF16 sink and recent pages instead.
// Per tile:
//  * S = K^ Q^T: A = the tile's K codes (rows = tokens = TMEM lanes), fed as the
//    fp16 subnormals c 4^p 2^-24 (p the code's position in its 16-bit half);
//    B = the query group's fragments q~ 2^sigma 4^-p as fp16 high and low parts,
//    16 columns (group, head, part); D = S (16 fp32 columns of TMEM).
//  * Token thread i reads its row of S, forms its 4 heads' logits with the
//    token's scale and zero and updates the online softmax with a lazy maximum
//    (O is rescaled in TMEM only when a head's maximum grows by more than 2^8,
//    so the weights stay below 2^8); it writes its weights p s_V 2^sigma_w as
//    fp16 high and low parts into the shared-memory B operand of the next
//    product and sums p and p z_V in fp32.
//  * O^T += V^ P^T: A = the tile's V codes (rows = channels = TMEM lanes) as
//    exact fp16 codes, B = the weights (16 columns: group, head, part), D = O^T
//    (16 fp32 columns of TMEM), accumulated over the split.
// Roles: warps 0-3 the tokens (K unpack, softmax, weights), warps 4-7 the
// channels (V unpack); thread 0 also issues the MMAs and the bulk copies of the
// page ring, right after the token warps' named barrier that follows each
// tile's K unpack (the barrier orders the K operand and the previous tile's
// weights before the MMAs that read them). The K operand is single-buffered,
// S and the V operand are double-buffered, the ring holds four tiles. Within a
// page, k position 2 (8 w + p) + e is token 16 (p >> 1) + 2 w + 8 (p & 1) + e,
// the order in which the channel-major V code words hold a channel's tokens. Every wait is bounded;
// a CTA whose wait expires flags OSCAR_STATUS_TIMEOUT and writes empty
// partials. Each history CTA writes one partial (m, l, acc[128]) per query head
// into slot `split`; the merge kernel combines the slots.
#include "bf16_page.cuh"
#include "kernels.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"
#include "timeline.cuh"

namespace oscar {
namespace {

constexpr int kTcThreads = 8 * 32;
constexpr int kTcStages = 4;                             // ring stages, one tile (two page blocks) each
constexpr int kTileTok = 2 * kP;                         // tokens per tile
constexpr int kStageBytes = 2 * kBlockBytes;             // 10,240
// B operands in shared memory, no swizzle, K-major: 8-row x 16-byte core matrices
constexpr int kQLbo = 128, kQSbo = (kD / 8) * kQLbo;     // S's B: 16 rows x 128 channel positions
constexpr int kPLbo = 144, kPSbo = (kTileTok / 8) * kPLbo;   // O's B: 16 rows x 128 token positions; the
                                                              // 144-byte K step keeps the token threads'
                                                              // 2-byte stores free of bank conflicts
constexpr int kQBytes = 2 * kQSbo;                       // 4,096
constexpr int kPBytes = 2 * kPSbo;                       // 4,608
constexpr int kOffQ = kTcStages * kStageBytes;           // 40,960
constexpr int kOffP = kOffQ + kQBytes;                   // two buffers
constexpr int kPidCap = 256;                             // page ids of a split held in shared memory
constexpr int kOffPid = kOffP + 2 * kPBytes;
constexpr int kOffRed = kOffPid + kPidCap * 4;           // [4 warps][16] floats, then [16] floats
constexpr int kOffBar = kOffRed + 5 * 16 * 4;
constexpr int kBFull = 0, kBEmpty = 4, kBSDone = 8, kBVFull = 10, kBODone = 12, kBFinal = 14, kNumBars = 15;
constexpr int kTcSmem = kOffBar + kNumBars * 8 + 16 + 1024;   // + TMEM address and flag, alignment slack
// TMEM (256 columns): the K operand, two V operands, two S tiles, O
constexpr uint32_t kTcCols = 256, kColAK = 0, kColAV = 64, kColS = 192, kColO = 224;
constexpr uint32_t kIdescN16 = idesc_f16(128, 16);
constexpr float kLazy = 8.f;                             // log2 growth of a maximum that forces a rescale
constexpr uint32_t kMagic = 0x64006400u;                 // fp16 1024.0 in both halves

__device__ __forceinline__ int canon_q(int n, int k) {
  return (n >> 3) * kQSbo + (k >> 3) * kQLbo + (n & 7) * 16 + (k & 7) * 2;
}
__device__ __forceinline__ int canon_p(int n, int k) {
  return (n >> 3) * kPSbo + (k >> 3) * kPLbo + (n & 7) * 16 + (k & 7) * 2;
}
// exact fp16 codes from (1024 + c 4^k): ((1024 + c 4^k) 4^-k) - 1024 4^-k = c, both halves
__device__ __forceinline__ uint32_t exact_codes(uint32_t biased, int k) {
  const uint32_t scale = 0x3C003C00u - (uint32_t)(k * 0x08000800u);
  const uint32_t offs = 0xE400E400u - (uint32_t)(k * 0x08000800u);
  return hfma2_u(biased, scale, offs);
}
__device__ __forceinline__ uint32_t half_bits(float x) { return (uint32_t)__half_as_ushort(__float2half_rn(x)); }
// OR of a predicate over the 128 threads of warps 0-3 (named barrier 1)
__device__ __forceinline__ bool tok_any(bool p) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred a, b;\n setp.ne.u32 a, %1, 0;\n bar.red.or.pred b, 1, 128, a;\n selp.u32 %0, 1, 0, b;\n}"
      : "=r"(r)
      : "r"((uint32_t)p)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void tok_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__global__ void __launch_bounds__(kTcThreads, 2) k_decode_tc(LayerView lv, DecodeWorkspace ws, FusedArgs fa) {
  TimelineSpan timeline_span(lv, kTlDecodeMma);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int h = blockIdx.y, b = blockIdx.z, split = blockIdx.x;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  pdl_launch_dependents();                         // the merge may be scheduled now; it waits for this grid
  if (split >= fa.nsplit) {                        // the BF16 pages of (b, h), one after another, warps 0-3
    if (w < 4) {
      for (int c = 0; c < fa.nbf; ++c) {
        bf16_page(lv, ws, fa, smem, c, h, b);
        bf16p::cta128_sync();                      // its shared memory is reused by the next page
      }
    }
    return;
  }

  const int gq = lv.hq / lv.hkv;
  uint8_t* ring = smem;
  const uint32_t bar0 = smem_addr(smem + kOffBar);
  auto BAR = [&](int k) { return bar0 + 8u * (uint32_t)k; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + kNumBars * 8);
  volatile int* failed = reinterpret_cast<volatile int*>(smem + kOffBar + kNumBars * 8 + 4);
  int* pid_s = reinterpret_cast<int*>(smem + kOffPid);
  float* red = reinterpret_cast<float*>(smem + kOffRed);

  // ---- pages of this split ------------------------------------------------------------------------------
  const int L = fa.seq_lens[b] + fa.len_add;
  int Lh = max(0, L - lv.sink - lv.recent);
  int npages = (Lh + kP - 1) / kP;
  if (npages > fa.max_hist_pages) {
    if (tid == 0 && split == 0) flag(lv.status, OSCAR_STATUS_BAD_SEQLEN);
    npages = fa.max_hist_pages;
    Lh = npages * kP;
  }
  const int nown = npages - fa.hist_start;
  if (nown < 0 && tid == 0 && split == 0) flag(lv.status, OSCAR_STATUS_BAD_SEQLEN);   // shorter than the shared prefix
  const int p0 = fa.hist_start + (int)((long long)split * max(nown, 0) / fa.nsplit);
  const int p1 = fa.hist_start + (int)((long long)(split + 1) * max(nown, 0) / fa.nsplit);
  const int np = p1 - p0, T = (np + 1) / 2;
  const int* pt = fa.hist_pt + (size_t)b * fa.max_hist_pages;
  auto page_id = [&](int k) -> int { return k < kPidCap ? pid_s[k] : __ldcg(pt + p0 + k); };
  // tile t into ring stage t % kTcStages (thread 0 only); false for a bad page id
  auto issue_tile = [&](int t) -> bool {
    const int s = t % kTcStages, n = min(2, np - 2 * t);
    int pid[2];
    for (int j = 0; j < n; ++j) {
      pid[j] = page_id(2 * t + j);
      if (pid[j] < 0 || pid[j] >= lv.n_int2) {
        flag(lv.status, OSCAR_STATUS_BAD_PAGE);
        return false;
      }
    }
    mbar_expect_tx(BAR(kBFull + s), (uint32_t)(n * kBlockBytes));
    const uint64_t pol = l2_evict_first();
    for (int j = 0; j < n; ++j)
      bulk_copy_hint(smem_addr(ring + s * kStageBytes + j * kBlockBytes), int2_block(lv, pid[j], h), kBlockBytes,
                     BAR(kBFull + s), pol);
    return true;
  };
  int issued = 0;                                  // tiles whose copies were issued (thread 0)
  if (w == 0) {
    for (int k = lane; k < np && k < kPidCap; k += 32) pid_s[k] = __ldcg(pt + p0 + k);
    __syncwarp();
    if (lane == 0) {
      for (int s = 0; s < kTcStages; ++s) {
        mbar_init_n(BAR(kBFull + s), 1);
        mbar_init_n(BAR(kBEmpty + s), 8);          // one arrival per token and channel warp
      }
      for (int j = 0; j < 2; ++j) {
        mbar_init_n(BAR(kBSDone + j), 1);
        mbar_init_n(BAR(kBVFull + j), 128);
        mbar_init_n(BAR(kBODone + j), 1);
      }
      mbar_init_n(BAR(kBFinal), 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      *failed = 0;
      // Before the programmatic wait only tiles the append cannot write are requested: it writes one row of
      // the request's last history page (the demoted token).
      while (issued < min(T, kTcStages) && p0 + 2 * issued + min(2, np - 2 * issued) - 1 < npages - 1) {
        if (!issue_tile(issued)) {
          *failed = 1;
          break;
        }
        ++issued;
      }
    }
    __syncwarp();
  }
  pdl_wait();                                      // q~, its constants and the appended row come from the prologue
  if (w == 0) {
    if (lane == 0 && !*failed) {
      for (; issued < min(T, kTcStages); ++issued)
        if (!issue_tile(issued)) {
          *failed = 1;
          break;
        }
    }
    __syncwarp();
    // Tensor memory is taken only after the wait: a CTA of this grid waiting above holds none, so a kernel
    // before it in the stream that allocates tensor memory (the shared-prefix decode) always can.
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kTcCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }

  // ---- the query fragments (S's B operand) and the weights' scale, token warps (thread = k position) ----
  float F[4], Z0[4], Z1[4];
  if (w < 4) {
    const int k = tid, c = k >> 1;
    const int p = c & 3, ch = 16 * (c >> 3) + 4 * ((c >> 2) & 1) + p + 8 * (k & 1), G = ch >> 6;
    uint8_t* qb = smem + kOffQ;
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      uint32_t hi = 0u, lo = 0u;
      F[hh] = Z0[hh] = Z1[hh] = 0.f;
      if (hh < gq) {
        const size_t row = (size_t)b * lv.hq + h * gq + hh;
        const float* qc = ws.qconst + row * kQConst;
        F[hh] = qc[kQF] * 16777216.f;              // 2^24: the key codes are fed as subnormals
        Z0[hh] = qc[kQZ0];
        Z1[hh] = qc[kQZ1];
        const int sig = (int)qc[kQSigma];
        const float x = ws.qrot[row * kD + ch] * exp2f((float)(sig - 2 * p));
        const float xh = frag_round16(x);
        hi = half_bits(xh);
        lo = half_bits(frag_round16(x - xh));
      }
      *reinterpret_cast<uint16_t*>(qb + canon_q(8 * G + 2 * hh, k)) = (uint16_t)hi;
      *reinterpret_cast<uint16_t*>(qb + canon_q(8 * G + 2 * hh + 1, k)) = (uint16_t)lo;
      *reinterpret_cast<uint16_t*>(qb + canon_q(8 * (1 - G) + 2 * hh, k)) = 0;
      *reinterpret_cast<uint16_t*>(qb + canon_q(8 * (1 - G) + 2 * hh + 1, k)) = 0;
    }
    // largest V clip threshold of this kv head: bounds every V scale, hence the weights' range
    float tv = fabsf(lv.params[(size_t)h * kParamFloats + kTauVOff + k]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tv = fmaxf(tv, __shfl_xor_sync(0xffffffffu, tv, o));
    if (lane == 0) red[64 + w] = tv;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the MMAs read the fragments
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // weights p s_V 2^sigma_w: p <= 2^8 and s_V <= max tau_V keep them below 2^15 (fp16-safe) and their low
  // parts clear of fp16 subnormals; O is scaled back by 2^-sigma_w
  int sigw = 0;
  {
    const float tmax = fmaxf(fmaxf(red[64], red[65]), fmaxf(red[66], red[67]));
    int e = 0;
    if (tmax > 0.f && tmax < INFINITY) frexpf(tmax, &e);
    sigw = min(max(7 - e, -60), 60);
  }
  const float wscale = exp2f((float)sigw);

  float mrun[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  float lsum[4] = {0.f, 0.f, 0.f, 0.f}, zs0[4] = {0.f, 0.f, 0.f, 0.f}, zs1[4] = {0.f, 0.f, 0.f, 0.f};
  bool ok = !*failed;
  if (w < 4) {
    // ================= token warps: thread = token i of the tile = TMEM lane i =================
    const int i = tid, pi = i >> 6, row = i & 63;
    // k position of this token: column 8 w + p of the V operand, w its V word and p its code position
    const int kpos = 64 * pi + 2 * (8 * v_word(row) + 2 * (row >> 4) + ((row >> 3) & 1)) + (row & 1);
    const uint32_t tl = tmem + ((uint32_t)(32 * w) << 16);
    auto unpack_k = [&](int t) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(BAR(kBFull + t % kTcStages), (t / kTcStages) & 1))) return false;
      const uint8_t* blk = ring + (t % kTcStages) * kStageBytes + pi * kBlockBytes + kKCodesOff + row * 32;
      const uint4 k0 = *reinterpret_cast<const uint4*>(blk), k1 = *reinterpret_cast<const uint4*>(blk + 16);
      const uint32_t wd[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t r[32];                            // column 8q + 4s + p: channels (16q + 4s + p, + 8), weight 4^p
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const uint32_t lo = wd[4 * half + qq], hi = lo >> 8;
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            r[8 * qq + p] = lo & (0x00030003u << (2 * p));
            r[8 * qq + 4 + p] = hi & (0x00030003u << (2 * p));
          }
        }
        tmem_st32u(tl + kColAK + 32 * half, r);
      }
      tmem_wait_st();
      tc_fence_before();
      return true;
    };
    // thread 0, after a named barrier of the token warps: S of tile t (its K operand is unpacked)
    const uint32_t qa = smem_addr(smem + kOffQ), pa = smem_addr(smem + kOffP);
    auto issue_s = [&](int t) {
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < 8; ++j)                  // channel positions 16 j .. 16 j + 15
        umma_ta(tmem + kColS + 16 * (t & 1), tmem + kColAK + 8 * j, umma_desc(qa + 2 * j * kQLbo, kQLbo, kQSbo),
                kIdescN16, j > 0);
      umma_commit(BAR(kBSDone + (t & 1)));
    };
    // thread 0, after a named barrier that follows the weights of tile t: O^T += V^ P^T once V is unpacked
    auto issue_o = [&](int t) -> bool {
      const int ab = t & 1;
      if (!mbar_wait(BAR(kBVFull + ab), (t >> 1) & 1)) return false;
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < 8; ++j)                  // tokens 16 j .. 16 j + 15 of the tile
        umma_ta(tmem + kColO, tmem + kColAV + 64 * ab + 8 * j,
                umma_desc(pa + ab * kPBytes + 2 * j * kPLbo, kPLbo, kPSbo), kIdescN16, t > 0 || j > 0);
      umma_commit(BAR(kBODone + ab));
      return true;
    };
    if (ok && T > 0) ok = unpack_k(0);
    if (tok_any(!ok)) ok = false;
    if (ok && T > 0 && tid == 0) issue_s(0);
    for (int t = 0; t < T && ok; ++t) {
      // S of this tile, and O of tile t - 2 done with this tile's weights buffer; the exits below are taken
      // by the four token warps together (they meet at named barrier 1)
      const int sb = t & 1;
      bool good = !*failed && mbar_wait(BAR(kBSDone + sb), (t >> 1) & 1);
      if (t >= 2) good = good && mbar_wait(BAR(kBODone + sb), ((t - 2) >> 1) & 1);
      good = __all_sync(0xffffffffu, good);
      uint32_t sr[16];
      if (good) {
        tc_fence_after();
        tmem_ld16(tl + kColS + 16 * sb, sr);
        tmem_wait_ld();
        if (t + 1 < T) good = unpack_k(t + 1);     // S(t) has read the K operand
      }
      if (tok_any(!good)) {
        ok = false;
        break;
      }
      if (tid == 0) {
        // the K operand of tile t + 1 and the weights of tile t - 1 are in: their MMAs, then the ring stage
        // of tile t - 1 takes tile t + 3
        bool fine = true;
        if (t + 1 < T) issue_s(t + 1);
        if (t >= 1) fine = issue_o(t - 1);
        if (fine && t >= 1 && t + kTcStages - 1 < T) {
          fine = mbar_wait(BAR(kBEmpty + (t - 1) % kTcStages), ((t - 1) / kTcStages) & 1) &&
                 issue_tile(t + kTcStages - 1);
          if (fine) issued = t + kTcStages;
        }
        if (!fine) *failed = 1;                    // seen by every token thread at its next barrier
      }
      // ---- logits of token i ----
      const int k = 2 * t + pi;
      const bool valid = k < np && (p0 + k) * kP + row < Lh;
      const uint8_t* blk = ring + (t % kTcStages) * kStageBytes + pi * kBlockBytes;
      const uint2 mk = *reinterpret_cast<const uint2*>(blk + kKMetaOff + row * 8);
      const uint2 mv = *reinterpret_cast<const uint2*>(blk + kVMetaOff + row * 8);
      const float2 ks0 = __half22float2(*reinterpret_cast<const __half2*>(&mk.x));   // (scale, zero), group 0
      const float2 ks1 = __half22float2(*reinterpret_cast<const __half2*>(&mk.y));
      float l[4];
      bool need = false;
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const float a0 = __uint_as_float(sr[2 * hh]) + __uint_as_float(sr[2 * hh + 1]);
        const float a1 = __uint_as_float(sr[8 + 2 * hh]) + __uint_as_float(sr[8 + 2 * hh + 1]);
        const float x = fmaf(F[hh], fmaf(ks0.x, a0, ks1.x * a1), fmaf(ks0.y, Z0[hh], ks1.y * Z1[hh]));
        l[hh] = (valid && hh < gq) ? x : -INFINITY;
        need |= l[hh] > mrun[hh] + kLazy;
      }
      if (tok_any(need)) {
        // a maximum grows by more than 2^8: the tile's maxima, then O, the sums and the maxima rescaled
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          float x = l[hh];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
          if (lane == 0) red[16 * w + hh] = x;
        }
        tok_sync();
        float f[4];
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          const float tm = fmaxf(fmaxf(red[hh], red[16 + hh]), fmaxf(red[32 + hh], red[48 + hh]));
          const float mn = fmaxf(mrun[hh], tm);
          f[hh] = (mrun[hh] == -INFINITY || mn == -INFINITY) ? (mrun[hh] == -INFINITY ? 0.f : 1.f)
                                                              : exp2f(mrun[hh] - mn);
          mrun[hh] = mn;
          lsum[hh] *= f[hh];
          zs0[hh] *= f[hh];
          zs1[hh] *= f[hh];
        }
        if (t > 0) {                               // O of tiles < t, complete, times the factors
          const bool got = __all_sync(0xffffffffu, mbar_wait(BAR(kBODone + ((t - 1) & 1)), ((t - 1) >> 1) & 1));
          if (tok_any(!got)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t o[16];
          tmem_ld16(tl + kColO, o);
          tmem_wait_ld();
#pragma unroll
          for (int n = 0; n < 16; ++n) o[n] = __float_as_uint(__uint_as_float(o[n]) * f[(n & 7) >> 1]);
          tmem_st16(tl + kColO, o);
          tmem_wait_st();
        }
        tok_sync();                                // every warp has read the tile maxima
      }
      // ---- weights ----
      const float2 vs0 = __half22float2(*reinterpret_cast<const __half2*>(&mv.x));   // (scale, zero), group 0
      const float2 vs1 = __half22float2(*reinterpret_cast<const __half2*>(&mv.y));
      float pw[4];
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        pw[hh] = (valid && hh < gq) ? fast_exp2(l[hh] - mrun[hh]) : 0.f;
        lsum[hh] += pw[hh];
        zs0[hh] = fmaf(pw[hh], valid ? vs0.y : 0.f, zs0[hh]);
        zs1[hh] = fmaf(pw[hh], valid ? vs1.y : 0.f, zs1[hh]);
      }
      uint8_t* pb = smem + kOffP + sb * kPBytes;
      const float sv0 = valid ? vs0.x * wscale : 0.f, sv1 = valid ? vs1.x * wscale : 0.f;
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
#pragma unroll
        for (int G = 0; G < 2; ++G) {
          const float x = pw[hh] * (G ? sv1 : sv0);
          const __half xh = __float2half_rn(x);
          *reinterpret_cast<uint16_t*>(pb + canon_p(8 * G + 2 * hh, kpos)) = __half_as_ushort(xh);
          *reinterpret_cast<uint16_t*>(pb + canon_p(8 * G + 2 * hh + 1, kpos)) =
              (uint16_t)half_bits(x - __half2float(xh));
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the MMAs read the weights
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(kBEmpty + t % kTcStages));      // the tile's codes and metadata are read
    }
    // O of the last tile, once every token warp's weights are in
    if (tok_any(!ok)) ok = false;
    if (ok && T > 0 && tid == 0 && !issue_o(T - 1)) *failed = 1;
    if (ok && T > 0 && !__all_sync(0xffffffffu, mbar_wait(BAR(kBODone + ((T - 1) & 1)), ((T - 1) >> 1) & 1)))
      ok = false;
    if (tid == 0) {
      if (!ok || *failed) {
        // copies still in flight land before the CTA leaves (bounded waits)
        for (int t = max(0, issued - kTcStages); t < issued; ++t)
          mbar_wait(BAR(kBFull + t % kTcStages), (t / kTcStages) & 1);
      }
      umma_commit(BAR(kBFinal));                   // every MMA completes before TMEM is read or released
      mbar_wait(BAR(kBFinal), 0);
    }
    // sums over the tokens: per warp, then through shared memory
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      float a = lsum[hh], z0 = zs0[hh], z1 = zs1[hh];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        z0 += __shfl_xor_sync(0xffffffffu, z0, o);
        z1 += __shfl_xor_sync(0xffffffffu, z1, o);
      }
      lsum[hh] = a;
      zs0[hh] = z0;
      zs1[hh] = z1;
    }
  } else if (w < 8) {
    // ================= channel warps: thread = channel c = TMEM lane c =================
    const int c = tid - 128;
    const uint32_t tl = tmem + ((uint32_t)(32 * (w - 4)) << 16);
    for (int t = 0; t < T && ok; ++t) {
      if (__any_sync(0xffffffffu, *failed != 0)) { ok = false; break; }
      const int s = t % kTcStages, ab = t & 1;
      bool got = mbar_wait(BAR(kBFull + s), (t / kTcStages) & 1);
      if (got && t >= 2) got = mbar_wait(BAR(kBODone + ab), ((t - 2) >> 1) & 1);   // O(t - 2) read this buffer
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int pi = 0; pi < 2; ++pi) {
        const uint4 v = *reinterpret_cast<const uint4*>(ring + s * kStageBytes + pi * kBlockBytes + v_chan_off(c));
        const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
        uint32_t r[32];                            // column 8w + p: the even and odd token of word w, position p
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const uint32_t lo = wd[qq], hi = lo >> 8;
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            r[8 * qq + p] = exact_codes(and_or(lo, 0x00030003u << (2 * p), kMagic), p);
            r[8 * qq + 4 + p] = exact_codes(and_or(hi, 0x00030003u << (2 * p), kMagic), p);
          }
        }
        tmem_st32u(tl + kColAV + 64 * ab + 32 * pi, r);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(kBEmpty + s));
      mbar_arrive(BAR(kBVFull + ab));
    }
  }
  __syncwarp();
  if (!ok) {
    if (!*failed) flag(lv.status, OSCAR_STATUS_TIMEOUT);
    *failed = 1;
  }
  // ---- partials: channel thread c writes channel c of every head -----------------------------------
  if (w < 4 && lane == 0) {
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      red[16 * w + hh] = lsum[hh];
      red[16 * w + 4 + hh] = zs0[hh];
      red[16 * w + 8 + hh] = zs1[hh];
      if (w == 0) red[64 + 8 + hh] = mrun[hh];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (w >= 4 && w < 8) {
    const int c = tid - 128, G = c >> 6;
    const bool live = !*failed && T > 0;
    float o[16] = {};
    if (live) {
      uint32_t r[16];
      tmem_ld16(tmem + ((uint32_t)(32 * (w - 4)) << 16) + kColO, r);
      tmem_wait_ld();
#pragma unroll
      for (int n = 0; n < 16; ++n) o[n] = __uint_as_float(r[n]);
    }
    const float unscale = exp2f((float)-sigw);
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      if (hh >= gq) break;
      float M = -INFINITY, Ls = 0.f, A = 0.f;
      if (live) {
        M = red[64 + 8 + hh];
        Ls = red[hh] + red[16 + hh] + red[32 + hh] + red[48 + hh];
        const int zo = G ? 8 : 4;
        const float Z = red[zo + hh] + red[16 + zo + hh] + red[32 + zo + hh] + red[48 + zo + hh];
        const float oc = G ? o[8 + 2 * hh] + o[9 + 2 * hh] : o[2 * hh] + o[2 * hh + 1];
        A = fmaf(oc, unscale, Z);
        if (M == -INFINITY) { Ls = 0.f; A = 0.f; }
      }
      float* part = part_row(ws, b, lv.hq, h * gq + hh, split);
      if (c == 0) {
        part[0] = M;
        part[1] = Ls;
      }
      part[4 + c] = A;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (w == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcCols) : "memory");
  }
}

}  // namespace

bool decode_tc_supported(const LayerView& lv) {
  return !lv.meta_u8 && !lv.meta_cb && lv.hq / lv.hkv <= 4;
}

int launch_decode_tc(const LayerView& lv, const DecodeWorkspace& ws, const DecodeArgs& a, float scale_log2,
                     cudaStream_t st) {
  FusedArgs fa = {};
  fa.seq_lens = a.seq_lens;
  fa.len_add = a.len_add;
  fa.hist_pt = a.hist_pt;
  fa.max_hist_pages = a.max_hist_pages;
  fa.nsplit = a.nsplit;
  fa.nbf = a.nbf;
  fa.hist_start = a.shared_pages;
  fa.bf_slot0 = a.nsplit + a.nsplit_shared;
  fa.bf16_pt = a.bf16_pt;
  fa.q = static_cast<const __nv_bfloat16*>(a.q);
  fa.scale_log2 = scale_log2;
  fa.out = a.out;
  fa.out_dtype = a.out_dtype;
  fa.lse = a.lse;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(a.nsplit + 1, lv.hkv, a.B);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTcSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode_tc, lv, ws, fa) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int configure_tc_kernel() {
  const void* f = reinterpret_cast<const void*>(k_decode_tc);
  if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem) != cudaSuccess)
    return OSCAR_ERR_CUDA;
  return set_max_shared_carveout(f);
}

}  // namespace oscar
