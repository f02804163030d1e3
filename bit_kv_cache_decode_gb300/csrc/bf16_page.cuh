// The BF16 sink + recent pages of the fused decode kernels (sm_103a): one page of
// 64 tokens per call, exact attention partial (m, l, acc) over its live rows.
//
// News article "超越 TurboQuant…OSCAR…", section "OSCAR 的设计思路": the BF16
// kernel handles the sink and recent windows; its partial is merged with the
// INT2 history's by the online-softmax merge. It runs on the first four warps
// (128 threads) of its CTA and synchronises them with named barrier 1, so a
// kernel with more warps can hand it one of its CTAs.
#pragma once

#include "kernels.cuh"
#include "tma.cuh"

namespace oscar {

struct FusedArgs {
  const int* seq_lens;
  int len_add;                       // attend over seq_lens[b] + len_add tokens
  const int* hist_pt;
  int max_hist_pages;
  int nsplit;                        // history CTAs per group
  int nbf;                           // BF16 pages per request
  int bf_fold;                       // > 0: the last nbf history CTAs also take one BF16 page each and give up
                                     // this many history pages for it; 0: the next nbf CTAs take one each
  int hist_start;                    // first history page of the splits (the pages before are shared ones)
  int bf_slot0;                      // partial slot of BF16 page 0
  const int* bf16_pt;
  const __nv_bfloat16* q;            // raw queries, for the BF16 tokens
  float scale_log2;                  // sm_scale * log2(e)
  void* out;
  int out_dtype;
  float* lse;
};

__device__ __forceinline__ float* part_row(const DecodeWorkspace& ws, int b, int hq_total, int hq, int slot) {
  return ws.partials + (((size_t)b * hq_total + hq) * ws.nslots + slot) * kPartFloats;
}

namespace bf16p {

// named barrier 1 over the 128 threads of warps 0-3
__device__ __forceinline__ void cta128_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool cta128_and(bool p) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred a, b;\n setp.ne.u32 a, %1, 0;\n bar.red.and.pred b, 1, 128, a;\n selp.u32 %0, 1, 0, b;\n}"
      : "=r"(r)
      : "r"((uint32_t)p)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(x));
  return d;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// p = hi + lo as two bf16 pairs (hi the rounded value, lo the rounded remainder), for (x, y)
__device__ __forceinline__ void split_bf16x2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x - __low2float(h), y - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

constexpr int kBfRow = kD + 8;       // bf16 per staged row: 272 bytes, so the 8 rows of an ldmatrix hit distinct banks
constexpr int kObStride = kD + 4;    // floats per (warp, head) row of the output combine

// BF16 page c of group (b, h): c = 0 is the sink page, c >= 1 the recent ring
// pages. Attention is order-independent, so each page is attended as a unit:
// row r is live if r < n_sink (sink page) or if its ring slot 64 (c - 1) + r <
// n_recent (ring pages). The live rows of K and V arrive by one bulk copy per
// row into padded rows (the rest are zero), and both products run on the
// tensor cores (mma.m16n8k16, bf16 in, f32 out), warp w taking tokens
// 16w .. 16w + 15:
//  * logits = K q^T: A = K rows (ldmatrix), B = the raw query rows of the
//    group's heads (8 columns, exact bf16 products);
//  * P.V: A = V^T (ldmatrix.trans), B = the weights as bf16 hi + lo parts (two
//    MMAs, so the weights keep about 16 bits), built from the logits'
//    accumulator layout by movmatrix transposes.
// The four warps' maxima, sums and outputs are combined through shared memory.
__device__ __forceinline__ void bf16_page(const LayerView& lv, const DecodeWorkspace& ws, const FusedArgs& fa,
                                          uint8_t* smem, int c, int h, int b) {
  __nv_bfloat16* ks = reinterpret_cast<__nv_bfloat16*>(smem);                   // [64][kBfRow]
  __nv_bfloat16* vs = ks + kP * kBfRow;                                         // [64][kBfRow]
  float* red = reinterpret_cast<float*>(vs + kP * kBfRow);                      // [2][4 warps][8 heads]
  float* ob = reinterpret_cast<float*>(smem);                                   // [4][8][kObStride], after the MMAs
  const uint32_t bar = smem_addr(red + 64);
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int gq = lv.hq / lv.hkv, hq0 = h * gq;
  pdl_wait();                                      // the append writes into these pages
  const int L = fa.seq_lens[b] + fa.len_add;
  if (L < 1 && tid == 0 && c == 0) flag(lv.status, OSCAR_STATUS_BAD_SEQLEN);
  const int n_sink = max(0, min(L, lv.sink));
  const int n_rec = L > lv.sink ? min(L - lv.sink, lv.recent) : 0;
  const int sink_pages = lv.sink / kP;
  int nrow;                                        // live rows are 0 .. nrow-1
  if (c < sink_pages) nrow = max(0, min(kP, n_sink - c * kP));
  else nrow = max(0, min(kP, n_rec - (c - sink_pages) * kP));
  const int page = nrow > 0 ? fa.bf16_pt[(size_t)b * ((lv.sink + lv.recent) / kP) + c] : -1;
  const bool ok = nrow > 0 && page >= 0 && page < lv.n_bf16;
  if (nrow > 0 && !ok && tid == 0) flag(lv.status, OSCAR_STATUS_BAD_PAGE);
  bool landed = false;
  uint32_t qb[8][2];                               // B fragments of the logits: head g, channels of k-step kk
  if (ok) {
    if (tid == 0) {
      mbar_init(bar);
      mbar_expect_tx(bar, 2u * nrow * kD * 2);
    }
    cta128_sync();                                 // barrier armed before any copy is issued
    {
      const int r = tid & (kP - 1), kind = tid >> 6;           // one row of K (kind 0) or V (kind 1) per thread
      __nv_bfloat16* dst = (kind ? vs : ks) + r * kBfRow;
      if (r < nrow) {
        const uint8_t* src = lv.bf16 + ((size_t)page * lv.hkv + h) * kBf16BlockBytes + ((size_t)kind * kP + r) * kD * 2;
        bulk_copy(smem_addr(dst), src, kD * 2, bar);
      } else {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int i = 0; i < kD / 8; ++i) d4[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    const __nv_bfloat16* qrow = fa.q + ((size_t)b * lv.hq + hq0 + g) * kD;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qb[kk][0] = g < gq ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * t) : 0u;
      qb[kk][1] = g < gq ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * t + 8) : 0u;
    }
    landed = cta128_and(mbar_wait(bar, 0));       // also publishes the zeroed rows
    if (!landed && tid == 0) flag(lv.status, OSCAR_STATUS_TIMEOUT);
  }
  if (!ok || !landed) {                            // block-uniform: nothing to attend (or the copy never came)
#pragma unroll
    for (int hh = 0; hh < 8; ++hh) {
      if (hh >= gq) break;
      float* part = part_row(ws, b, lv.hq, hq0 + hh, fa.bf_slot0 + c);
      if (tid == 0) { part[0] = -INFINITY; part[1] = 0.f; }
      part[4 + tid] = 0.f;
    }
    return;
  }
  // ---- logits of tokens 16w + g (s[0], s[1]) and 16w + g + 8 (s[2], s[3]), heads 2t, 2t + 1 ----
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const uint32_t ka = smem_addr(ks) + ((16 * w + (lane & 7) + 8 * ((lane >> 3) & 1)) * kBfRow + 8 * (lane >> 4)) * 2;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(ka + kk * 32, a0, a1, a2, a3);
      mma_bf16(s, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
    }
  }
  const int tok0 = 16 * w + g, tok1 = tok0 + 8;
#pragma unroll
  for (int e = 0; e < 4; ++e) s[e] = ((e < 2 ? tok0 : tok1) < nrow) ? s[e] * fa.scale_log2 : -INFINITY;
  // ---- maxima and sums per head over the page ------------------------------------------------------
  float m0 = fmaxf(s[0], s[2]), m1 = fmaxf(s[1], s[3]);
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, x));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, x));
  }
  if (g == 0) { red[w * 8 + 2 * t] = m0; red[w * 8 + 2 * t + 1] = m1; }
  cta128_sync();
  float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
  for (int ww = 0; ww < 4; ++ww) { M0 = fmaxf(M0, red[ww * 8 + 2 * t]); M1 = fmaxf(M1, red[ww * 8 + 2 * t + 1]); }
  float p[4];
  p[0] = M0 == -INFINITY ? 0.f : fast_exp2(s[0] - M0);
  p[1] = M1 == -INFINITY ? 0.f : fast_exp2(s[1] - M1);
  p[2] = M0 == -INFINITY ? 0.f : fast_exp2(s[2] - M0);
  p[3] = M1 == -INFINITY ? 0.f : fast_exp2(s[3] - M1);
  float l0 = p[0] + p[2], l1 = p[1] + p[3];
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, x);
    l1 += __shfl_xor_sync(0xffffffffu, l1, x);
  }
  if (g == 0) { red[32 + w * 8 + 2 * t] = l0; red[32 + w * 8 + 2 * t + 1] = l1; }
  // ---- P.V over the warp's 16 tokens, all 128 channels ------------------------------------------------
  uint32_t bh0, bl0, bh1, bl1;
  split_bf16x2(p[0], p[1], bh0, bl0);              // tokens 16w + g: heads 2t, 2t + 1
  split_bf16x2(p[2], p[3], bh1, bl1);              // tokens 16w + g + 8
  bh0 = movmatrix_t(bh0); bl0 = movmatrix_t(bl0);  // head g, tokens 2t, 2t + 1
  bh1 = movmatrix_t(bh1); bl1 = movmatrix_t(bl1);  // head g, tokens 2t + 8, 2t + 9
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  {
    const uint32_t va = smem_addr(vs) + ((16 * w + (lane & 7) + 8 * (lane >> 4)) * kBfRow + 8 * ((lane >> 3) & 1)) * 2;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(va + mt * 32, a0, a1, a2, a3);     // channels 16 mt .., tokens 16 w ..
      mma_bf16(o[mt], a0, a1, a2, a3, bh0, bh1);
      mma_bf16(o[mt], a0, a1, a2, a3, bl0, bl1);
    }
  }
  cta128_sync();                                   // every warp's K / V reads are done: ob may overwrite them
  // o[mt]: channel 16 mt + g (0, 1) or + 8 (2, 3), head 2t (0, 2) or 2t + 1 (1, 3)
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    float* r0 = ob + (w * 8 + 2 * t) * kObStride + 16 * mt + g;
    r0[0] = o[mt][0];
    r0[kObStride] = o[mt][1];
    r0[8] = o[mt][2];
    r0[kObStride + 8] = o[mt][3];
  }
  cta128_sync();
#pragma unroll
  for (int hh = 0; hh < 8; ++hh) {
    if (hh >= gq) break;
    float M = -INFINITY, Ls = 0.f, A = 0.f;
#pragma unroll
    for (int ww = 0; ww < 4; ++ww) {
      M = fmaxf(M, red[ww * 8 + hh]);
      Ls += red[32 + ww * 8 + hh];
      A += ob[(ww * 8 + hh) * kObStride + tid];
    }
    float* part = part_row(ws, b, lv.hq, hq0 + hh, fa.bf_slot0 + c);
    if (tid == 0) { part[0] = M; part[1] = Ls; }
    part[4 + tid] = A;
  }
  // the copies have landed: the barrier is retired, so that a later call may set up another one here
  if (tid == 0) asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

}  // namespace bf16p

using bf16p::bf16_page;

}  // namespace oscar
