// All-BF16 paged decode (sm_103a): the comparison kernel, the same attention
// over a plain BF16 paged cache (news article "超越 TurboQuant…OSCAR…",
// section "系统加速效果", and MarkTechPost article "Together AI 开源 OSCAR…",
// section "结果": OSCAR's decode speed-up is measured against a BF16 KV cache).
//
// Work: grid (split, kv head, request), 128 threads (4 warps). A CTA streams
// the pages of its split through a 3-stage ring: a page block (K [64][128]
// then V [64][128] bf16, 32 KB) arrives by 128 row copies (cp.async.bulk, one
// row per thread) into rows padded to 272 bytes, so the eight rows of every
// ldmatrix sit in distinct banks; rows past the sequence end are zero-filled.
// Warp w takes tokens 16 w .. 16 w + 15 of every page:
//  * logits = K q^T on the tensor cores (mma.m16n8k16, bf16 in, f32 out), A =
//    the K rows (ldmatrix), B = the raw bf16 queries of the group (column =
//    query head, exact products);
//  * an online softmax over the warp's tokens (running maximum and sum per
//    head, the output rescaled when the maximum grows);
//  * O^T += V^T P, A = V^T (ldmatrix.trans), B = the weights as bf16 high and
//    low parts (two MMAs, about 16 bits of weight).
// The four warps' (m, l, acc) combine at the end into one partial per query
// head; k_merge_plain merges the splits.
#include "kernels.cuh"
#include "tma.cuh"

namespace oscar {
namespace {

constexpr int kStages = 3;
constexpr int kRow = kD + 8;                        // bf16 per staged row: 272 bytes
constexpr int kStageHalves = 2 * kP * kRow;         // K rows then V rows
constexpr int kStreamSmem = kStages * kStageHalves * 2 + kStages * 8 + 16 + 128;

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(x));
  return d;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// (x, y) as bf16 high parts and the rounded remainders
__device__ __forceinline__ void split_hi_lo(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x - __low2float(h), y - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__global__ void __launch_bounds__(128, 2) k_bf16_stream(const uint8_t* __restrict__ pages, int hkv, int hq_total,
                                                       int num_pages, const __nv_bfloat16* __restrict__ q,
                                                       const int* __restrict__ seq_lens,
                                                       const int* __restrict__ page_table, int max_pages,
                                                       int pages_per_split, float scale_log2,
                                                       float* __restrict__ partials, int nslots, int* status) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __nv_bfloat16* ring = reinterpret_cast<__nv_bfloat16*>(smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u));
  const uint32_t bar0 = smem_addr(ring + kStages * kStageHalves);
  __shared__ float cm[4][8], cl[4][8];
  // the warps' output accumulators [4][8][kD + 4] take the ring's place once the pages are consumed
  float (*co)[8][kD + 4] = reinterpret_cast<float (*)[8][kD + 4]>(ring);
  static_assert(4 * 8 * (kD + 4) * 4 <= kStages * kStageHalves * 2, "combine buffer fits the ring");
  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int gq = hq_total / hkv, hq0 = h * gq;
  int L = seq_lens[b];
  if (L > max_pages * kP || L < 1) {
    if (tid == 0 && s == 0) flag(status, OSCAR_STATUS_BAD_SEQLEN);
    L = max(0, min(L, max_pages * kP));
  }
  const int npages = (L + kP - 1) / kP;
  const int p0 = min(npages, s * pages_per_split), p1 = min(npages, (s + 1) * pages_per_split);
  const int n = p1 - p0;
  const int* pt = page_table + (size_t)b * max_pages;
  if (tid == 0) {
    for (int k = 0; k < kStages; ++k) mbar_init(bar0 + 8 * k);
  }
  __syncthreads();
  // page k of the split into stage k % kStages: thread r copies row r (K rows 0..63, then V rows), rows past
  // the sequence end (and every row of a bad page) are zero-filled; thread 0 announces the bytes
  const uint64_t pol = l2_evict_first();
  auto issue = [&](int k) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // after the generic reads of the stage
    const int page = pt[p0 + k];
    const bool ok = page >= 0 && page < num_pages;
    if (!ok && tid == 0) flag(status, OSCAR_STATUS_BAD_PAGE);
    const int nrow = ok ? min(kP, L - (p0 + k) * kP) : 0;
    const uint32_t bar = bar0 + 8 * (k % kStages);
    if (tid == 0) mbar_expect_tx(bar, (uint32_t)(2 * nrow * kD * 2));
    const int r = tid & (kP - 1), kind = tid >> 6;
    __nv_bfloat16* dst = ring + (k % kStages) * kStageHalves + (kind * kP + r) * kRow;
    if (r < nrow) {
      const uint8_t* src = pages + ((size_t)page * hkv + h) * kBf16BlockBytes + ((size_t)kind * kP + r) * kD * 2;
      bulk_copy_hint(smem_addr(dst), src, kD * 2, bar, pol);
    } else {
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int i = 0; i < kD / 8; ++i) d4[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  int issued = 0;
  for (; issued < kStages && issued < n; ++issued) issue(issued);
  // B fragments of the logits: head g (columns past the group are zero), channels of k-step kk
  uint32_t qb[8][2];
  {
    const __nv_bfloat16* qrow = q + ((size_t)b * hq_total + hq0 + g) * kD;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qb[kk][0] = g < gq ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * t) : 0u;
      qb[kk][1] = g < gq ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * t + 8) : 0u;
    }
  }
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // heads 2t, 2t + 1
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  bool good = true;
  for (int k = 0; k < n; ++k) {
    const int st = k % kStages;
    good = __syncthreads_and(mbar_wait(bar0 + 8 * st, (k / kStages) & 1));   // also: zero-filled rows visible
    if (!good) {
      if (tid == 0) flag(status, OSCAR_STATUS_TIMEOUT);
      break;
    }
    const __nv_bfloat16* ks = ring + st * kStageHalves;
    const __nv_bfloat16* vs = ks + kP * kRow;
    // logits of tokens 16 w + g (s[0], s[1]) and 16 w + g + 8 (s[2], s[3]), heads 2t, 2t + 1
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const uint32_t ka = smem_addr(ks) + ((16 * w + (lane & 7) + 8 * ((lane >> 3) & 1)) * kRow + 8 * (lane >> 4)) * 2;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t a[4];
        ldsm4(ka + kk * 32, a);
        mma_bf16(sc, a, qb[kk][0], qb[kk][1]);
      }
    }
    const int tok = (p0 + k) * kP + 16 * w + g;
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[e] = (tok + 8 * (e >> 1) < L) ? sc[e] * scale_log2 : -INFINITY;
    float x0 = fmaxf(sc[0], sc[2]), x1 = fmaxf(sc[1], sc[3]);
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, x));
      x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, x));
    }
    const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
    if (n0 > m0 || n1 > m1) {                      // the running maxima grow: rescale this lane's heads
      const float a0 = m0 == -INFINITY ? 0.f : ex2(m0 - n0), a1 = m1 == -INFINITY ? 0.f : ex2(m1 - n1);
      l0 *= a0;
      l1 *= a1;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= a0;
        o[mt][2] *= a0;
        o[mt][1] *= a1;
        o[mt][3] *= a1;
      }
      m0 = n0;
      m1 = n1;
    }
    float p[4];
    p[0] = m0 == -INFINITY ? 0.f : ex2(sc[0] - m0);
    p[1] = m1 == -INFINITY ? 0.f : ex2(sc[1] - m1);
    p[2] = m0 == -INFINITY ? 0.f : ex2(sc[2] - m0);
    p[3] = m1 == -INFINITY ? 0.f : ex2(sc[3] - m1);
    l0 += p[0] + p[2];
    l1 += p[1] + p[3];
    // P.V over the warp's 16 tokens, all 128 channels
    uint32_t bh0, bl0, bh1, bl1;
    split_hi_lo(p[0], p[1], bh0, bl0);             // token 16w + g: heads 2t, 2t + 1
    split_hi_lo(p[2], p[3], bh1, bl1);             // token 16w + g + 8
    bh0 = movmatrix_trans(bh0);                    // head g, tokens 2t, 2t + 1
    bl0 = movmatrix_trans(bl0);
    bh1 = movmatrix_trans(bh1);                    // head g, tokens 2t + 8, 2t + 9
    bl1 = movmatrix_trans(bl1);
    {
      const uint32_t va = smem_addr(vs) + ((16 * w + (lane & 7) + 8 * (lane >> 4)) * kRow + 8 * ((lane >> 3) & 1)) * 2;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t a[4];
        ldsm4_t(va + mt * 32, a);                  // channels 16 mt .., tokens 16 w ..
        mma_bf16(o[mt], a, bh0, bh1);
        mma_bf16(o[mt], a, bl0, bl1);
      }
    }
    __syncthreads();                               // every warp is done with this stage
    if (k + kStages < n) {
      issue(k + kStages);
      ++issued;
    }
  }
  if (!good) {                                     // the copies in flight land before the ring is reused (bounded)
    for (int k = max(0, issued - kStages); k < issued; ++k) mbar_wait(bar0 + 8 * (k % kStages), (k / kStages) & 1);
  }
  __syncthreads();
  // combine the warps: per head, maximum, sum and the channel accumulators
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, x);
    l1 += __shfl_xor_sync(0xffffffffu, l1, x);
  }
  if (g == 0) {
    cm[w][2 * t] = m0;
    cm[w][2 * t + 1] = m1;
    cl[w][2 * t] = l0;
    cl[w][2 * t + 1] = l1;
  }
  // o[mt]: channel 16 mt + g (0, 1) or + 8 (2, 3), head 2t (0, 2) or 2t + 1 (1, 3)
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    co[w][2 * t][16 * mt + g] = o[mt][0];
    co[w][2 * t + 1][16 * mt + g] = o[mt][1];
    co[w][2 * t][16 * mt + g + 8] = o[mt][2];
    co[w][2 * t + 1][16 * mt + g + 8] = o[mt][3];
  }
  __syncthreads();
  for (int hh = 0; hh < gq; ++hh) {
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < 4; ++ww) M = fmaxf(M, cm[ww][hh]);
    float Ls = 0.f, A = 0.f;
    if (M != -INFINITY && good) {
#pragma unroll
      for (int ww = 0; ww < 4; ++ww) {
        if (cm[ww][hh] == -INFINITY) continue;
        const float f = ex2(cm[ww][hh] - M);
        Ls = fmaf(cl[ww][hh], f, Ls);
        A = fmaf(co[ww][hh][tid], f, A);
      }
    } else {
      M = -INFINITY;
    }
    float* part = partials + (((size_t)b * hq_total + hq0 + hh) * nslots + s) * kPartFloats;
    if (tid == 0) {
      part[0] = M;
      part[1] = Ls;
    }
    part[4 + tid] = A;
  }
}

}  // namespace

int launch_bf16_stream(int B, int hkv, int hq, const void* kv_pages, int num_pages, const void* q,
                       const int* seq_lens, const int* page_table, int max_pages, int pages_per_split, int nsplit,
                       float scale_log2, float* partials, int nslots, int* status, cudaStream_t st) {
  k_bf16_stream<<<dim3(nsplit, hkv, B), 128, kStreamSmem, st>>>(
      static_cast<const uint8_t*>(kv_pages), hkv, hq, num_pages, static_cast<const __nv_bfloat16*>(q), seq_lens,
      page_table, max_pages, pages_per_split, scale_log2, partials, nslots, status);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int configure_bf16_stream() {
  return cudaFuncSetAttribute(k_bf16_stream, cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamSmem) ==
                 cudaSuccess
             ? OSCAR_OK
             : OSCAR_ERR_CUDA;
}

}  // namespace oscar
