// Shared-prefix history decode on the tensor cores (sm_103a).
//
// MarkTechPost article "Together AI 开源 OSCAR…", section "服务系统：混合精度缓存
// 布局": the pool stays compatible with paged KV and prefix caching, so requests
// of a batch that share a prompt prefix share its history pages through their
// page tables. This kernel reads each shared page once per step for all the
// batch's queries of a kv head, instead of once per request.
//
// Work: grid (split, kv head, query tile); 8 warps. A CTA takes the shared
// pages [p0, p1) of its split and the query tile's 128 query rows (request r,
// head i flattened as r * gq + i), warp w owning rows 16 w .. 16 w + 15.
//  * Each page (5120 B block: K codes | V codes | K meta | V meta) arrives by
//    one bulk copy in a 3-stage ring. The CTA expands it once into shared
//    memory: K as the fp16 numbers 1024 + 256 c (every code moved into mantissa
//    bits 8-9, so the constant part is 4x the code term at most), V as its
//    exact codes c. Page i + 1 is expanded while page i is consumed
//    (double-buffered).
//  * Logits: mma.m16n8k16 with A = K rows (ldmatrix), B = fragments of the
//    warp's queries (q~ 2^sigma / 256 as fp16 high + low parts, one column
//    each), one accumulator per channel group started from minus the
//    fragments' 1024 * sum, then scale / zero per token and group as in the
//    per-request kernel.
//  * P.V: A = the V codes transposed (rows = channels; ldmatrix), B = the
//    weights times the token's V scale of the tile's channel group (fp16),
//    built from the logits' accumulator layout with movmatrix transposes; the
//    zero-point part sum_t p_t z_t is accumulated in fp32 per group, as in the
//    per-request kernel.
// Each CTA writes one partial (m, l, acc[128]) per query row into the history
// slot `slot0 + split`; the merge kernel combines it with the request's other
// slots.
#include "kernels.cuh"
#include "tma.cuh"
#include "timeline.cuh"

namespace oscar {
namespace {

constexpr int kShWarps = 8;
constexpr int kShThreads = kShWarps * 32;
constexpr int kShQ = 16 * kShWarps;                   // query rows per CTA
static_assert(kShQ == kSharedRows, "the host's query tiles");
constexpr int kShStages = 3;
constexpr int kKhStride = kD + 8;                     // fp16 per expanded K row: 272 B
constexpr int kVtStride = kP + 8;                     // fp16 per expanded V^T row: 144 B
constexpr int kKhBytes = kP * kKhStride * 2;          // 17,408
constexpr int kVtBytes = kD * kVtStride * 2;          // 18,432
constexpr int kShFragWords = kShWarps * 8 * 4 * 32 * 2;   // [warp][k-block][n-tile][lane][2]: 64 KB
// per query row: F, the fragment scale 2^sigma / 256, Z0, Z1, and the offsets 1024 sum(high + low) of
// channel groups 0 and 1; the pairs read as float2 sit at even indices
constexpr int kShConst = 8;
constexpr int kCF = 0, kCScale = 1, kCZ = 2, kCOff = 4;
constexpr uint32_t kMagic = 0x64006400u;              // fp16 1024.0 in both halves
constexpr uint32_t kCodeMask = 0x03000300u;           // mantissa bits 8-9 of both halves

// shared-memory layout (bytes)
constexpr int kOffRing = 0;
constexpr int kOffKh = kOffRing + kShStages * kBlockBytes;          // 2 buffers
constexpr int kOffVt = kOffKh + 2 * kKhBytes;                       // 2 buffers
constexpr int kOffFrag = kOffVt + 2 * kVtBytes;
constexpr int kOffConst = kOffFrag + kShFragWords * 4;
constexpr int kOffBar = kOffConst + kShQ * kShConst * 4;
constexpr int kShSmem = kOffBar + kShStages * 8 + 8 + 128;          // + a timeout flag, + alignment slack
static_assert(kShQ * kD * 4 <= 2 * kKhBytes + 2 * kVtBytes, "q~ staging fits in the expansion buffers");

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(x));
  return d;
}

__device__ __forceinline__ uint32_t and_or(uint32_t x, uint32_t mask, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "r"(mask), "r"(magic));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
  const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b),
                            *reinterpret_cast<const __half2*>(&c));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// fp16 rounding of a fragment value, subnormal results flushed to zero
__device__ __forceinline__ float frag_round16(float x) {
  const float r = __half2float(__float2half_rn(x));
  return fabsf(r) < 6.103515625e-05f ? 0.f : r;
}

// The 2-bit code i (bits 2i) of both 16-bit halves of x, moved to bits 8-9 and fed as fp16
// 1024 + 256 c (i is a compile-time constant after unrolling).
__device__ __forceinline__ uint32_t code_at(uint32_t x, int i) {
  const uint32_t y = i < 4 ? (x << (8 - 2 * i)) : (x >> (2 * i - 8));
  return and_or(y, kCodeMask, kMagic);
}

// Expanded V^T: row = channel; the fp16 pair of tokens (2p, 2p+1) sits in 16-byte chunk (p / 4) ^ ((row / 8) % 8)
// of the row, word p % 4. The 8 rows an ldmatrix reads share one swizzle (conflict-free with the padded rows),
// the expansion's stores spread over the banks, and an ldmatrix address is a per-lane base plus a constant.
__device__ __forceinline__ int vt_word(int row, int p) {
  return row * (kVtStride / 2) + 4 * ((p >> 2) ^ ((row >> 3) & 7)) + (p & 3);
}


// Expand one packed page block into the K and V^T buffers (all threads; 2 K words and 2 V words each).
__device__ __forceinline__ void expand_page(const uint8_t* blk, __half* kh, uint32_t* vt) {
#pragma unroll
  for (int k2 = 0; k2 < 2; ++k2) {
    const int wi = threadIdx.x + kShThreads * k2;              // 0 .. 511
    {                                                          // K: token tk, channels 16 u .. 16 u + 15
      const int tk = wi >> 3, u = wi & 7;
      const uint32_t x = *reinterpret_cast<const uint32_t*>(blk + kKCodesOff + tk * 32 + 4 * u);
      // fp16 pair r_i = (channel 16u + i, channel 16u + 8 + i) goes to positions 2i, 2i + 1 of the block
      uint4* dst = reinterpret_cast<uint4*>(kh + tk * kKhStride + 16 * u);
      dst[0] = make_uint4(code_at(x, 0), code_at(x, 1), code_at(x, 2), code_at(x, 3));
      dst[1] = make_uint4(code_at(x, 4), code_at(x, 5), code_at(x, 6), code_at(x, 7));
    }
    {                                                          // V: tokens 2p, 2p + 1, channels 8 o .. 8 o + 7
      const int p = wi >> 4, o = wi & 15;
      const uint32_t x = *reinterpret_cast<const uint32_t*>(blk + kVCodesOff + p * 64 + 4 * o);
#pragma unroll
      for (int i = 0; i < 8; ++i)                              // the exact codes: (1024 + 256 c) / 256 - 4 = c
        vt[vt_word(8 * o + i, p)] = hfma2_u(code_at(x, i), 0x1C001C00u, 0xC400C400u);
    }
  }
}

struct SharedArgs {
  const int* hist_pt;                // [B][max_hist_pages]; the shared prefix is read from request 0's row
  int shared_pages;                  // history pages [0, shared_pages) are the same for every request
  int nsplit;                        // shared splits per kv head
  int slot0;                         // partial slot of split 0
  int B;
};

__global__ void __launch_bounds__(kShThreads, 1) k_decode_shared(LayerView lv, DecodeWorkspace ws, SharedArgs sa) {
  TimelineSpan timeline_span(lv, kTlDecodeShared);
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
  __shared__ int page_ok[kShStages];
  const int split = blockIdx.x, h = blockIdx.y, qt = blockIdx.z;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int gq = lv.hq / lv.hkv, nq = sa.B * gq;
  uint8_t* ring = smem + kOffRing;
  uint32_t* frag_s = reinterpret_cast<uint32_t*>(smem + kOffFrag);
  float* qc_s = reinterpret_cast<float*>(smem + kOffConst);
  const uint32_t bar0 = smem_addr(smem + kOffBar);

  const int np = sa.shared_pages;
  const int p0 = (int)((long long)split * np / sa.nsplit);
  const int n = (int)((long long)(split + 1) * np / sa.nsplit) - p0;
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kShStages; ++s) mbar_init(bar0 + 8 * s);
  }
  __syncthreads();
  // page k of the split into stage k % 3 (thread 0); the step prologue never writes shared pages, so
  // the first ones are requested before the programmatic wait
  int issued_n = 0;                                // pages requested so far (thread 0)
  auto issue = [&](int k) {
    issued_n = k + 1;
    const int pid = __ldcg(sa.hist_pt + p0 + k);
    const bool ok = pid >= 0 && pid < lv.n_int2;
    if (ok) {
      bulk_load_hint(smem_addr(ring + (k % kShStages) * kBlockBytes), int2_block(lv, pid, h), kBlockBytes,
                     bar0 + 8 * (k % kShStages), l2_evict_first());
    } else {
      flag(lv.status, OSCAR_STATUS_BAD_PAGE);
    }
    page_ok[k % kShStages] = ok;
  };
  if (tid == 0) {
    for (int k = 0; k < kShStages && k < n; ++k) issue(k);
  }
  pdl_launch_dependents();
  pdl_wait();                                      // q~ and its constants come from the step prologue

  // ---- the tile's query rows: q~ staged in the expansion buffers, then fragments and constants ----
  float* qs = reinterpret_cast<float*>(smem + kOffKh);          // [kShQ][kD]
  for (int e = tid; e < kShQ * kD / 4; e += kShThreads) {
    const int ql = e / (kD / 4), c4 = e % (kD / 4), Q = qt * kShQ + ql;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (Q < nq) {
      const int r = Q / gq, hq = h * gq + Q % gq;
      v = *reinterpret_cast<const float4*>(ws.qrot + ((size_t)r * lv.hq + hq) * kD + 4 * c4);
    }
    reinterpret_cast<float4*>(qs)[e] = v;
  }
  __syncthreads();
  // per row (warp w: rows w, w + 8, ...): F, Z0, Z1 and the fragment offsets 1024 * sum(part) per group
  for (int ql = w; ql < kShQ; ql += kShWarps) {
    const int Q = qt * kShQ + ql;
    float F = 0.f, Z0 = 0.f, Z1 = 0.f, sig = 0.f;
    if (Q < nq) {
      const float* qc = ws.qconst + ((size_t)(Q / gq) * lv.hq + h * gq + Q % gq) * kQConst;
      F = qc[kQF];
      Z0 = qc[kQZ0];
      Z1 = qc[kQZ1];
      sig = qc[kQSigma];
    }
    const float sc = exp2f(sig - 8.f);             // fragment value x = q~ 2^sigma / 256
    float offh = 0.f, offl = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {                  // lane l: channels 4l .. 4l + 3 (group l / 16)
      const float x = qs[ql * kD + 4 * lane + e] * sc;
      const float hi = frag_round16(x);
      offh += hi;
      offl += frag_round16(x - hi);
    }
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) {
      offh += __shfl_xor_sync(0xffffffffu, offh, m);
      offl += __shfl_xor_sync(0xffffffffu, offl, m);
    }
    if (lane == 0) {
      qc_s[ql * kShConst + kCF] = F;
      qc_s[ql * kShConst + kCScale] = sc;
      qc_s[ql * kShConst + kCZ] = Z0;
      qc_s[ql * kShConst + kCZ + 1] = Z1;
    }
    if (lane == 0 || lane == 16) qc_s[ql * kShConst + kCOff + (lane >> 4)] = 1024.f * offh + 1024.f * offl;
  }
  __syncthreads();
  // B fragments: word (warp ww, k-block kb, n-tile nb, part, lane (g', t'), r) holds, for row
  // 16 ww + 8 nb + g' and its high (part 0) or low (part 1) fp16 parts, the channels at k rows 2t' + 8r
  // and 2t' + 8r + 1 of the k-block: 16 kb + t' + 4r and 16 kb + 8 + t' + 4r (the expanded K rows hold
  // channel i of a 16-channel block at position 2i, channel 8 + i at 2i + 1). Both parts accumulate
  // into the same column.
  for (int wi = tid; wi < kShFragWords; wi += kShThreads) {
    const int r = wi & 1, lp = (wi >> 1) & 31, part = (wi >> 6) & 1, nb = (wi >> 7) & 1, kb = (wi >> 8) & 7,
              ww = wi >> 11;
    const int ql = 16 * ww + 8 * nb + (lp >> 2), tp = lp & 3;
    const float sc = qc_s[ql * kShConst + kCScale];
    const int c0 = 16 * kb + tp + 4 * r;
    float x[2] = {qs[ql * kD + c0] * sc, qs[ql * kD + c0 + 8] * sc};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float hi = frag_round16(x[e]);
      x[e] = part ? frag_round16(x[e] - hi) : hi;
    }
    frag_s[wi] = pack_f16x2(x[0], x[1]);
  }
  __syncthreads();
  // the lane's 4 query rows j = 2 nb + e: row 16 w + 8 nb + 2t + e (n-tile nb, accumulator column 2t + e)
  auto qrow = [&](int j) { return 16 * w + 8 * (j >> 1) + 2 * t + (j & 1); };
  float cF[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) cF[j] = qc_s[qrow(j) * kShConst + kCF];
  __syncthreads();                                 // q~ staging is done: the buffers take pages now

  // ---- running state: vacc[b][mt] = channels 16 mt + g (+ 8), rows 8b + 2t (+ 1) --------------------
  float vacc[2][8][4];
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) vacc[b][mt][e] = 0.f;
  float mrun[4], lsum[4], zacc[4][2];             // zacc[j][G]: sum of p z over the lane's tokens, group G
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    mrun[j] = -INFINITY;
    lsum[j] = 0.f;
    zacc[j][0] = zacc[j][1] = 0.f;
  }
  bool timed_out = false;
  auto wait_page = [&](int k) {                    // every thread; page k was issued if page_ok says so
    const int s = k % kShStages;
    if (page_ok[s] && !mbar_wait(bar0 + 8 * s, (k / kShStages) & 1)) timed_out = true;
  };
  auto kh_of = [&](int buf) { return reinterpret_cast<__half*>(smem + kOffKh + buf * kKhBytes); };
  auto vt_of = [&](int buf) { return reinterpret_cast<uint32_t*>(smem + kOffVt + buf * kVtBytes); };
  if (n > 0) {
    wait_page(0);
    if (page_ok[0] && !timed_out) expand_page(ring, kh_of(0), vt_of(0));
  }
  timed_out = __syncthreads_or(timed_out);

  for (int i = 0; i < n && !timed_out; ++i) {
    const int s = i % kShStages, s1 = (i + 1) % kShStages;
    const bool ok_i = page_ok[s];
    if (i + 1 < n) {                               // expand page i + 1 while page i is consumed
      wait_page(i + 1);
      if (page_ok[s1] && !timed_out) expand_page(ring + s1 * kBlockBytes, kh_of((i + 1) & 1), vt_of((i + 1) & 1));
    }
    if (ok_i) {
      const uint8_t* blk = ring + s * kBlockBytes;
      const uint32_t kh_a = smem_addr(kh_of(i & 1)), vt_a = smem_addr(vt_of(i & 1));
      // this lane's ldmatrix row of V^T (vrow = lane % 8 + 8 hr) and chunk parity (token half h)
      const int hr = (lane >> 3) & 1, hh = lane >> 4;
      const uint32_t vt_lane = vt_a + ((lane & 7) + 8 * hr) * kVtStride * 2 + 16 * (hh ^ hr);
      // ---- logits of the page's 64 tokens for the warp's 16 rows -----------------------------------
      float lg[4][4][2];                           // [token tile m][query j][token 16m + g, 16m + g + 8]
#pragma unroll 1
      for (int G = 0; G < 2; ++G) {
        uint32_t bq[4][2][2][2];                   // [k-block 4G + kk][n-tile][part][reg]
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
          for (int nb = 0; nb < 2; ++nb)
#pragma unroll
            for (int pt = 0; pt < 2; ++pt) {
              const uint2 v = *reinterpret_cast<const uint2*>(
                  frag_s + (((((w * 8 + 4 * G + kk) * 2 + nb) * 2 + pt) * 32 + lane) * 2));
              bq[kk][nb][pt][0] = v.x;
              bq[kk][nb][pt][1] = v.y;
            }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          float acc[2][4];                         // n-tile nb: rows 8 nb + 2t (0, 2), + 1 (1, 3)
#pragma unroll
          for (int nb = 0; nb < 2; ++nb) {
            const float o0 = qc_s[qrow(2 * nb) * kShConst + kCOff + G];
            const float o1 = qc_s[qrow(2 * nb + 1) * kShConst + kCOff + G];
            acc[nb][0] = acc[nb][2] = -o0;
            acc[nb][1] = acc[nb][3] = -o1;
          }
          const uint32_t arow = kh_a + ((16 * m + (lane & 7) + 8 * ((lane >> 3) & 1)) * kKhStride + 8 * (lane >> 4)) * 2;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(arow + (16 * (4 * G + kk)) * 2, a0, a1, a2, a3);
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
              mma16816(acc[nb], a0, a1, a2, a3, bq[kk][nb][0][0], bq[kk][nb][0][1]);   // high parts
              mma16816(acc[nb], a0, a1, a2, a3, bq[kk][nb][1][0], bq[kk][nb][1][1]);   // low parts
            }
          }
          const uint2 mk0 = *reinterpret_cast<const uint2*>(blk + kKMetaOff + (16 * m + g) * 8);
          const uint2 mk1 = *reinterpret_cast<const uint2*>(blk + kKMetaOff + (16 * m + g + 8) * 8);
          const float2 sz0 = __half22float2(*reinterpret_cast<const __half2*>(G == 0 ? &mk0.x : &mk0.y));
          const float2 sz1 = __half22float2(*reinterpret_cast<const __half2*>(G == 0 ? &mk1.x : &mk1.y));
          if (G == 0) {
            const float2 zz0 = __half22float2(*reinterpret_cast<const __half2*>(&mk0.y));   // group 1 of row g
            const float2 zz1 = __half22float2(*reinterpret_cast<const __half2*>(&mk1.y));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 zc = *reinterpret_cast<const float2*>(qc_s + qrow(j) * kShConst + kCZ);   // Z0, Z1
              lg[m][j][0] = fmaf(cF[j] * sz0.x, acc[j >> 1][j & 1], fmaf(sz0.y, zc.x, zz0.y * zc.y));
              lg[m][j][1] = fmaf(cF[j] * sz1.x, acc[j >> 1][2 + (j & 1)], fmaf(sz1.y, zc.x, zz1.y * zc.y));
            }
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              lg[m][j][0] = fmaf(cF[j] * sz0.x, acc[j >> 1][j & 1], lg[m][j][0]);
              lg[m][j][1] = fmaf(cF[j] * sz1.x, acc[j >> 1][2 + (j & 1)], lg[m][j][1]);
            }
          }
        }
      }
      // ---- online softmax update (shared pages are full: all 64 tokens are live) -------------------
      float mref[4];
      bool grow = false;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float mx = -INFINITY;
#pragma unroll
        for (int m = 0; m < 4; ++m) mx = fmaxf(mx, fmaxf(lg[m][j][0], lg[m][j][1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        mref[j] = fmaxf(mrun[j], mx);
        grow |= mref[j] > mrun[j];
      }
      if (__any_sync(0xffffffffu, grow)) {
        float al[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          al[j] = mref[j] > mrun[j] ? exp2f(mrun[j] - mref[j]) : 1.f;
          lsum[j] *= al[j];
          zacc[j][0] *= al[j];
          zacc[j][1] *= al[j];
          mrun[j] = mref[j];
        }
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            vacc[b][mt][0] *= al[2 * b];
            vacc[b][mt][2] *= al[2 * b];
            vacc[b][mt][1] *= al[2 * b + 1];
            vacc[b][mt][3] *= al[2 * b + 1];
          }
      }
      // ---- P.V over the page's four 16-token tiles --------------------------------------------------
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        // V scale and zero of tokens 16 kt + g (x: group 0, y: group 1) and 16 kt + g + 8
        const uint2 mv0 = *reinterpret_cast<const uint2*>(blk + kVMetaOff + (16 * kt + g) * 8);
        const uint2 mv1 = *reinterpret_cast<const uint2*>(blk + kVMetaOff + (16 * kt + g + 8) * 8);
        const float2 v00 = __half22float2(*reinterpret_cast<const __half2*>(&mv0.x));   // (s, z), token g, group 0
        const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&mv0.y));   // group 1
        const float2 v10 = __half22float2(*reinterpret_cast<const __half2*>(&mv1.x));   // token g + 8
        const float2 v11 = __half22float2(*reinterpret_cast<const __half2*>(&mv1.y));
        float p[4][2];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          p[j][0] = fast_exp2(lg[kt][j][0] - mrun[j]);
          p[j][1] = fast_exp2(lg[kt][j][1] - mrun[j]);
          lsum[j] += p[j][0] + p[j][1];
          zacc[j][0] = fmaf(p[j][0], v00.y, fmaf(p[j][1], v10.y, zacc[j][0]));
          zacc[j][1] = fmaf(p[j][0], v01.y, fmaf(p[j][1], v11.y, zacc[j][1]));
        }
        uint32_t b0[2][2], b1[2][2];                  // [b][G]
#pragma unroll
        for (int b = 0; b < 2; ++b) {                 // row 8b + g, tokens 2t, 2t + 1 (b0) and 2t + 8, 2t + 9 (b1)
          b0[b][0] = movmatrix_t(pack_f16x2(p[2 * b][0] * v00.x, p[2 * b + 1][0] * v00.x));
          b1[b][0] = movmatrix_t(pack_f16x2(p[2 * b][1] * v10.x, p[2 * b + 1][1] * v10.x));
          b0[b][1] = movmatrix_t(pack_f16x2(p[2 * b][0] * v01.x, p[2 * b + 1][0] * v01.x));
          b1[b][1] = movmatrix_t(pack_f16x2(p[2 * b][1] * v11.x, p[2 * b + 1][1] * v11.x));
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {               // channels 16 mt ..: group mt / 4
          // row 16 mt + vrow, token pairs 8 kt + 4h ..: chunk (2 kt + h) ^ (2 (mt % 4) + hr) = 2 (kt ^ mt % 4) + (h ^ hr)
          uint32_t a0, a1, a2, a3;
          ldsm_x4(vt_lane + 16 * mt * kVtStride * 2 + 32 * (kt ^ (mt & 3)), a0, a1, a2, a3);
#pragma unroll
          for (int b = 0; b < 2; ++b) mma16816(vacc[b][mt], a0, a1, a2, a3, b0[b][mt >> 2], b1[b][mt >> 2]);
        }
      }
    }
    timed_out = __syncthreads_or(timed_out);      // page i's buffers and ring stage are free
    if (!timed_out && tid == 0 && i + kShStages < n) issue(i + kShStages);
  }

  if (timed_out) {
    // give the copies still in flight a bounded chance to land before the CTA's memory is released
    if (tid == 0) {                                // only the last use of each stage can be outstanding
      flag(lv.status, OSCAR_STATUS_TIMEOUT);
      for (int k = max(0, issued_n - kShStages); k < issued_n; ++k)
        if (page_ok[k % kShStages]) mbar_wait(bar0 + 8 * (k % kShStages), (k / kShStages) & 1);
    }
  }
  // ---- partials: one slot per query row ----------------------------------------------------------------
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      lsum[j] += __shfl_xor_sync(0xffffffffu, lsum[j], x);
      zacc[j][0] += __shfl_xor_sync(0xffffffffu, zacc[j][0], x);
      zacc[j][1] += __shfl_xor_sync(0xffffffffu, zacc[j][1], x);
    }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int Q = qt * kShQ + qrow(j);
    if (Q >= nq) continue;
    float* part = ws.partials + (((size_t)(Q / gq) * lv.hq + h * gq + Q % gq) * ws.nslots + sa.slot0 + split) *
                                    kPartFloats;
    const bool live = !timed_out && mrun[j] != -INFINITY;
    if (g == 0) {
      part[0] = live ? mrun[j] : -INFINITY;
      part[1] = live ? lsum[j] : 0.f;
    }
    const int b = j >> 1, e0 = j & 1;              // vacc elements e0 (channel 16mt + g), e0 + 2 (+ 8)
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const float zs = zacc[j][mt >> 2];
      part[4 + 16 * mt + g] = live ? vacc[b][mt][e0] + zs : 0.f;
      part[4 + 16 * mt + g + 8] = live ? vacc[b][mt][e0 + 2] + zs : 0.f;
    }
  }
}

}  // namespace

int launch_decode_shared(const LayerView& lv, const DecodeWorkspace& ws, const DecodeArgs& a, cudaStream_t st) {
  if (a.shared_pages <= 0 || a.nsplit_shared <= 0 || a.B == 0) return OSCAR_OK;
  SharedArgs sa;
  sa.hist_pt = a.hist_pt;
  sa.shared_pages = a.shared_pages;
  sa.nsplit = a.nsplit_shared;
  sa.slot0 = a.nsplit;
  sa.B = a.B;
  const int nq = a.B * (lv.hq / lv.hkv);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(a.nsplit_shared, lv.hkv, (nq + kShQ - 1) / kShQ);
  cfg.blockDim = dim3(kShThreads);
  cfg.dynamicSmemBytes = kShSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode_shared, lv, ws, sa) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int configure_shared_kernel() {
  if (cudaFuncSetAttribute(k_decode_shared, cudaFuncAttributeMaxDynamicSharedMemorySize, kShSmem) != cudaSuccess)
    return OSCAR_ERR_CUDA;
  return set_max_shared_carveout(reinterpret_cast<const void*>(k_decode_shared));
}

}  // namespace oscar
