// INT2 history decode on the tensor cores (sm_103a).
//
// News article "超越 TurboQuant…OSCAR…", section "OSCAR 的设计思路": the INT2
// kernel unpacks the 2-bit codes, restores scale/zero and accumulates in
// floating point; MarkTechPost article "Together AI 开源 OSCAR…", section "服务
// 系统：混合精度缓存布局": packed codes, per-token groups of 64 channels.
//
// Work: grid (split, kv head, request); 4 warps per CTA; warp w takes history
// pages p0 + w, p0 + w + 4, ... of the CTA's split. Each (page, kv head) block
// (5120 B: K codes | V codes | K meta | V meta) is copied into a per-warp
// 3-stage shared-memory ring by one cp.async.bulk with an mbarrier; waits are
// bounded and report OSCAR_STATUS_TIMEOUT instead of hanging.
//
// Per 16-token tile the two contractions run on mma.sync.m16n8k16 f16 -> f32:
//  * logits: A = codes [16 tokens x 16 channels], B = query fragments
//    [16 channels x 8 columns], column = (head, group) of a 4-head n-tile; the
//    code c of channel ch is fed as the fp16 value 1024 + c*4^(ch%4) (one
//    LOP3: mask | 0x6400), whose constant part and scale the query prologue
//    folded into the fragments and the per-head offsets;
//  * P.Vhat: A = codes [16 channels x 16 tokens] (the V page layout pairs two
//    tokens in one 32-bit word, so mask | 0x6400 and one HFMA2 give the exact
//    fp16 codes of one channel for two tokens), B = p * scale [16 tokens x 8
//    columns], built from the logits' accumulator layout with two movmatrix
//    transposes; the zero-point part sum_t p_t z_t is accumulated in fp32.
// The kernel ends with a combine of the 4 warps' online-softmax partials and
// writes one partial (m, l, acc[128]) per query head and split.
#include "kernels.cuh"

namespace oscar {

namespace {

constexpr int kWarps = 4;
constexpr int kStages = 3;
constexpr unsigned kWaitLimit = 1u << 24;
constexpr uint32_t kMagic = 0x64006400u;       // fp16 1024.0 in both halves
// stage ring, mbarriers, a timeout flag, and slack to align the ring to 128 bytes
constexpr int kMmaSmem = kWarps * kStages * kBlockBytes + kWarps * kStages * 8 + 16 + 128;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Bounded wait for the phase with the given parity; false when the limit expires.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (unsigned i = 0; i < kWaitLimit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
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

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// exact fp16 codes: ((1024 + c*4^k) * 4^-k) - 1024*4^-k = c, for both halves
__device__ __forceinline__ uint32_t exact_codes(uint32_t biased, int k) {
  const uint32_t scale = 0x3C003C00u - (uint32_t)(k * 0x08000800u);   // 4^-k = 2^-2k: exponent - 2k
  const uint32_t offs = 0xE400E400u - (uint32_t)(k * 0x08000800u);    // -1024 * 4^-k
  __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&biased), *reinterpret_cast<const __half2*>(&scale),
                      *reinterpret_cast<const __half2*>(&offs));
  return *reinterpret_cast<const uint32_t*>(&r);
}

template <int NT>
__global__ void __launch_bounds__(128, NT == 1 ? 3 : 2)
    k_int2_mma(LayerView lv, DecodeWorkspace ws, const int* __restrict__ seq_lens, const int* __restrict__ hist_pt,
               int max_hist_pages, int pages_per_split) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
  int& any_timeout = *reinterpret_cast<int*>(smem + kWarps * kStages * kBlockBytes + kWarps * kStages * 8);
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int gq = lv.hq / lv.hkv;
  if (tid == 0) any_timeout = 0;
  __syncthreads();

  // ---- pages of this warp --------------------------------------------------------
  const int L = seq_lens[b];
  int Lh = max(0, L - lv.sink - lv.recent);
  int npages = (Lh + kP - 1) / kP;
  if (npages > max_hist_pages) {
    if (tid == 0 && split == 0) flag(lv.status, OSCAR_STATUS_BAD_SEQLEN);
    npages = max_hist_pages;
    Lh = npages * kP;
  }
  const int p0 = split * pages_per_split + w;
  const int p1 = min(split * pages_per_split + pages_per_split, npages);
  const int my_pages = p0 < p1 ? (p1 - p0 + kWarps - 1) / kWarps : 0;
  const int* pt = hist_pt + (size_t)b * max_hist_pages;

  uint8_t* stage0 = smem + (size_t)w * kStages * kBlockBytes;
  const uint32_t stage_s = smem_addr(stage0);
  const uint32_t bar_s = smem_addr(smem + kWarps * kStages * kBlockBytes) + w * kStages * 8;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(bar_s + 8 * s);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  // issue the load of the warp's i-th page into stage i % kStages; returns whether it was issued
  auto issue = [&](int i) -> bool {
    const int page = p0 + kWarps * i;
    const int pid = pt[page];
    if (pid < 0 || pid >= lv.n_int2) {
      if (lane == 0) flag(lv.status, OSCAR_STATUS_BAD_PAGE);
      return false;
    }
    if (lane == 0) {
      const int s = i % kStages;
      bulk_load(stage_s + s * kBlockBytes, int2_block(lv, pid, h), kBlockBytes, bar_s + 8 * s);
    }
    return true;
  };
  uint32_t issued = 0;                 // bit s: a load is outstanding in stage s
#pragma unroll
  for (int i = 0; i < kStages; ++i)
    if (i < my_pages && issue(i)) issued |= 1u << i;

  // ---- per-lane constants -------------------------------------------------------
  uint32_t qf[8][NT][2];
  {
    const uint32_t* frag = ws.qfrag + ((size_t)b * lv.hkv + h) * kFragWords;
#pragma unroll
    for (int kb = 0; kb < 8; ++kb)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint2 v = *reinterpret_cast<const uint2*>(frag + ((kb * 2 + nt) * 32 + lane) * 2);
        qf[kb][nt][0] = v.x;
        qf[kb][nt][1] = v.y;
      }
  }
  float cF[NT], cZ0[NT], cZ1[NT], cO0[NT], cO1[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int head = 4 * nt + t;
    cF[nt] = cZ0[nt] = cZ1[nt] = cO0[nt] = cO1[nt] = 0.f;
    if (head < gq) {
      const float* qc = ws.qconst + ((size_t)b * lv.hq + h * gq + head) * kQConst;
      cF[nt] = qc[kQF];
      cZ0[nt] = qc[kQZ0];
      cZ1[nt] = qc[kQZ1];
      cO0[nt] = qc[kQOff0];
      cO1[nt] = qc[kQOff1];
    }
  }

  // ---- running state ----------------------------------------------------------------
  float acc[NT][8][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][mt][e] = 0.f;
  float mrun[NT], lsum[NT], zacc[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    mrun[nt] = -INFINITY;
    lsum[nt] = 0.f;
    zacc[nt][0] = zacc[nt][1] = 0.f;
  }
  uint32_t phase = 0;
  bool timed_out = false;

  for (int i = 0; i < my_pages; ++i) {
    const int s = i % kStages;
    if (issued & (1u << s)) {
      const bool landed = __all_sync(0xffffffffu, mbar_wait(bar_s + 8 * s, (phase >> s) & 1u));
      if (!landed) {                   // warp-uniform decision: the shuffles and MMAs below need every lane
        timed_out = true;
        break;
      }
      phase ^= 1u << s;
      issued &= ~(1u << s);
      const uint8_t* blk = stage0 + s * kBlockBytes;
      const int ntok = min(kP, Lh - (p0 + kWarps * i) * kP);

      // ---- logits of the page's 64 tokens -----------------------------------------
      float lg[4][NT][2];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int r0 = 16 * mt + g, r1 = r0 + 8;
        const uint2 kw0 = *reinterpret_cast<const uint2*>(blk + kKCodesOff + r0 * 32 + 8 * t);
        const uint2 kw1 = *reinterpret_cast<const uint2*>(blk + kKCodesOff + r1 * 32 + 8 * t);
        const uint32_t x0h = kw0.x >> 8, x1h = kw0.y >> 8, y0h = kw1.x >> 8, y1h = kw1.y >> 8;
        float c[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          const uint32_t m = 0x00030003u << (2 * (kb & 3));
          const uint32_t a0 = ((kb < 4 ? kw0.x : x0h) & m) | kMagic;
          const uint32_t a1 = ((kb < 4 ? kw1.x : y0h) & m) | kMagic;
          const uint32_t a2 = ((kb < 4 ? kw0.y : x1h) & m) | kMagic;
          const uint32_t a3 = ((kb < 4 ? kw1.y : y1h) & m) | kMagic;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816(c[nt], a0, a1, a2, a3, qf[kb][nt][0], qf[kb][nt][1]);
        }
        const uint2 mk0 = *reinterpret_cast<const uint2*>(blk + kKMetaOff + r0 * 8);
        const uint2 mk1 = *reinterpret_cast<const uint2*>(blk + kKMetaOff + r1 * 8);
        const float2 sz00 = __half22float2(*reinterpret_cast<const __half2*>(&mk0.x));   // scale0, zero0 of row r0
        const float2 sz01 = __half22float2(*reinterpret_cast<const __half2*>(&mk0.y));   // scale1, zero1
        const float2 sz10 = __half22float2(*reinterpret_cast<const __half2*>(&mk1.x));
        const float2 sz11 = __half22float2(*reinterpret_cast<const __half2*>(&mk1.y));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float l0 = fmaf(sz00.x, c[nt][0] - cO0[nt], sz01.x * (c[nt][1] - cO1[nt]));
          float l1 = fmaf(sz10.x, c[nt][2] - cO0[nt], sz11.x * (c[nt][3] - cO1[nt]));
          l0 = fmaf(cF[nt], l0, fmaf(sz00.y, cZ0[nt], sz01.y * cZ1[nt]));
          l1 = fmaf(cF[nt], l1, fmaf(sz10.y, cZ0[nt], sz11.y * cZ1[nt]));
          lg[mt][nt][0] = r0 < ntok ? l0 : -INFINITY;
          lg[mt][nt][1] = r1 < ntok ? l1 : -INFINITY;
        }
      }

      // ---- online softmax update ------------------------------------------------------
      float mnew[NT];
      bool grow = false;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float mx = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) mx = fmaxf(mx, fmaxf(lg[mt][nt][0], lg[mt][nt][1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        mnew[nt] = fmaxf(mrun[nt], mx);
        grow |= mnew[nt] > mrun[nt];
      }
      if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float al = (mnew[nt] > mrun[nt]) ? exp2f(mrun[nt] - mnew[nt]) : 1.f;
          lsum[nt] *= al;
          zacc[nt][0] *= al;
          zacc[nt][1] *= al;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][mt][e] *= al;
          mrun[nt] = mnew[nt];
        }
      }

      // ---- P.Vhat over the page's four 16-token tiles -----------------------------------
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        const int r0 = 16 * kt + g, r1 = r0 + 8;
        const uint2 mv0 = *reinterpret_cast<const uint2*>(blk + kVMetaOff + r0 * 8);
        const uint2 mv1 = *reinterpret_cast<const uint2*>(blk + kVMetaOff + r1 * 8);
        float2 sv00 = __half22float2(*reinterpret_cast<const __half2*>(&mv0.x));
        float2 sv01 = __half22float2(*reinterpret_cast<const __half2*>(&mv0.y));
        float2 sv10 = __half22float2(*reinterpret_cast<const __half2*>(&mv1.x));
        float2 sv11 = __half22float2(*reinterpret_cast<const __half2*>(&mv1.y));
        if (r0 >= ntok) sv00 = sv01 = make_float2(0.f, 0.f);       // rows past the end: no stale metadata
        if (r1 >= ntok) sv10 = sv11 = make_float2(0.f, 0.f);
        uint32_t bf[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float pa = exp2f(lg[kt][nt][0] - mrun[nt]);
          const float pb = exp2f(lg[kt][nt][1] - mrun[nt]);
          lsum[nt] += pa + pb;
          zacc[nt][0] = fmaf(pa, sv00.y, fmaf(pb, sv10.y, zacc[nt][0]));
          zacc[nt][1] = fmaf(pa, sv01.y, fmaf(pb, sv11.y, zacc[nt][1]));
          bf[nt][0] = movmatrix_t(pack_f16x2(pa * sv00.x, pa * sv01.x));
          bf[nt][1] = movmatrix_t(pack_f16x2(pb * sv10.x, pb * sv11.x));
        }
        const uint2 wab = *reinterpret_cast<const uint2*>(blk + kVCodesOff + (8 * kt + t) * 64 + 8 * g);
        const uint2 wcd = *reinterpret_cast<const uint2*>(blk + kVCodesOff + (8 * kt + t + 4) * 64 + 8 * g);
        const uint32_t wah = wab.x >> 8, wbh = wab.y >> 8, wch = wcd.x >> 8, wdh = wcd.y >> 8;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int k = mt & 3;
          const uint32_t m = 0x00030003u << (2 * k);
          const uint32_t a0 = exact_codes(((mt < 4 ? wab.x : wah) & m) | kMagic, k);   // channel 16g + mt, tokens 2t, 2t+1
          const uint32_t a1 = exact_codes(((mt < 4 ? wab.y : wbh) & m) | kMagic, k);   // channel 16g + 8 + mt
          const uint32_t a2 = exact_codes(((mt < 4 ? wcd.x : wch) & m) | kMagic, k);   // tokens 2t + 8, 2t + 9
          const uint32_t a3 = exact_codes(((mt < 4 ? wcd.y : wdh) & m) | kMagic, k);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt][mt], a0, a1, a2, a3, bf[nt][0], bf[nt][1]);
        }
      }
    }
    __syncwarp();
    const int next = i + kStages;
    if (next < my_pages && issue(next)) issued |= 1u << s;
  }

  if (timed_out) {
    // give the copies still in flight a bounded chance to land before the buffers are reused
    if (lane == 0) flag(lv.status, OSCAR_STATUS_TIMEOUT);
    for (int s = 0; s < kStages; ++s)
      if (issued & (1u << s)) mbar_wait(bar_s + 8 * s, (phase >> s) & 1u);
    any_timeout = 1;
  }

  // ---- reduce per-lane sums over the 8 lanes of a head, then combine the warps ---------
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      lsum[nt] += __shfl_xor_sync(0xffffffffu, lsum[nt], x);
      zacc[nt][0] += __shfl_xor_sync(0xffffffffu, zacc[nt][0], x);
      zacc[nt][1] += __shfl_xor_sync(0xffffffffu, zacc[nt][1], x);
    }
  }
  __syncthreads();
  float* cm = reinterpret_cast<float*>(smem);     // [kWarps][8] running max
  float* cl = cm + kWarps * 8;                    // [kWarps][8] running sum
  float* ca = cl + kWarps * 8;                    // [kWarps][8][128] accumulators
  const int grp = g >> 2;                         // channels 16g .. 16g+15 lie in group g / 4
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int head = 4 * nt + t;
    if (g == 0) {
      cm[w * 8 + head] = mrun[nt];
      cl[w * 8 + head] = lsum[nt];
    }
    const float zs = grp ? zacc[nt][1] : zacc[nt][0];
    float* dst = ca + (w * 8 + head) * kD;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      dst[16 * g + mt] = (grp ? acc[nt][mt][1] : acc[nt][mt][0]) + zs;
      dst[16 * g + 8 + mt] = (grp ? acc[nt][mt][3] : acc[nt][mt][2]) + zs;
    }
  }
  __syncthreads();
  const int nslots = ws.max_splits + 1;
  for (int hh = 0; hh < gq; ++hh) {
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, cm[ww * 8 + hh]);
    float Ls = 0.f, A = 0.f;
    if (M != -INFINITY && !any_timeout) {
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) {
        const float mw = cm[ww * 8 + hh];
        if (mw == -INFINITY) continue;
        const float f = exp2f(mw - M);
        Ls = fmaf(cl[ww * 8 + hh], f, Ls);
        A = fmaf(ca[(ww * 8 + hh) * kD + tid], f, A);
      }
    } else {
      M = -INFINITY;
    }
    float* part = ws.partials + (((size_t)b * lv.hq + h * gq + hh) * nslots + split) * kPartFloats;
    if (tid == 0) {
      part[0] = M;
      part[1] = Ls;
    }
    part[4 + tid] = A;
  }
}

}  // namespace

int launch_int2_mma(const LayerView& lv, const DecodeWorkspace& ws, const DecodeArgs& a, float, cudaStream_t st) {
  const dim3 grid(a.nsplit, lv.hkv, a.B);
  if (lv.hq / lv.hkv <= 4)
    k_int2_mma<1><<<grid, 128, kMmaSmem, st>>>(lv, ws, a.seq_lens, a.hist_pt, a.max_hist_pages, a.pages_per_split);
  else
    k_int2_mma<2><<<grid, 128, kMmaSmem, st>>>(lv, ws, a.seq_lens, a.hist_pt, a.max_hist_pages, a.pages_per_split);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int configure_mma_kernels() {
  if (cudaFuncSetAttribute(k_int2_mma<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmem) != cudaSuccess)
    return OSCAR_ERR_CUDA;
  if (cudaFuncSetAttribute(k_int2_mma<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmem) != cudaSuccess)
    return OSCAR_ERR_CUDA;
  return OSCAR_OK;
}

}  // namespace oscar
