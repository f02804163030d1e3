// INT2 history decode on the tensor cores (sm_103a).
//
// News article "超越 TurboQuant…OSCAR…", section "OSCAR 的设计思路": the INT2
// kernel unpacks the 2-bit codes, restores scale/zero and accumulates in
// floating point; MarkTechPost article "Together AI 开源 OSCAR…", section "服务
// 系统：混合精度缓存布局": packed codes, per-token groups of 64 channels.
//
// Work: grid (split, kv head, request); 4 warps per CTA; warp w takes history
// pages p0 + w, p0 + w + 4, ... of the CTA's split, a request's pages being
// spread evenly over the splits. Each (page, kv head) block
// (5120 B: K codes | V codes | K meta | V meta) is copied into a per-warp
// 2-stage shared-memory ring by one cp.async.bulk with an mbarrier; waits are
// bounded and report OSCAR_STATUS_TIMEOUT instead of hanging.
//
// Per 16-token tile the two contractions run on mma.sync.m16n8k16 f16 -> f32:
//  * logits: A = codes [16 tokens x 16 channels of one group], B = query
//    fragments [16 channels x 8 columns], column = (head, hi or lo fp16 part
//    of the query) of a 4-head n-tile, one accumulator per channel group; the
//    code c at bit position 2p of a 16-bit half is masked in place (one AND)
//    and fed as the fp16 subnormal c 4^(p mod 4) 2^-24; the query prologue
//    folded 4^-(p mod 4) and a power of two 2^sigma into the fragments (which
//    keeps the products clear of the subnormal range) and the logit scale
//    takes back 2^24 (codebook pools feed 1024 + k_c and subtract per-head
//    offsets instead);
//  * P.Vhat: A = codes [16 channels x 16 tokens] (the V page layout pairs two
//    tokens in one 32-bit word, so one AND gives the codes of one channel for
//    two tokens, as fp16 subnormals c 4^pos 2^-24 like the keys'), B = p *
//    scale * 4^-pos * 2^sw [16 tokens x 8 columns], sw a per-head power of two
//    from the largest V clip threshold, built from the logits' accumulator
//    layout with two movmatrix transposes; the zero-point part sum_t p_t z_t is
//    accumulated in fp32. Codebook pools feed their levels exactly instead.
// A history CTA ends with a combine of its 4 warps' online-softmax partials
// and writes one partial (m, l, acc[128]) per query head and split.
//
// The same launch carries the BF16 sink + recent tokens (row-wise bulk copies,
// tensor-core products), folded into the last history splits or as one extra
// CTA per BF16 page. The log-sum-exp merge of all slots runs as the next
// kernel (merge.cu), a programmatic dependent that is scheduled while this
// grid runs and waits for its completion.
#include "kernels.cuh"
#include "bf16_page.cuh"
#include "rotate.cuh"
#include "tma.cuh"
#include "timeline.cuh"

namespace oscar {

namespace {

constexpr int kWarps = 4;
constexpr int kStages = 2;                     // pages per warp: one in use, one in flight
constexpr float kLag = 8.f;                     // the softmax reference may lag the maximum by 2^kLag
// stage ring, mbarriers, a timeout flag, per warp the float32 metadata rows of its current page
// ([K, V][64 rows] x (scale, zero of group 0, scale, zero of group 1)), and slack to align to 128 bytes
constexpr int kMeta32Off = kWarps * kStages * kBlockBytes + kWarps * kStages * 8 + 16;
constexpr int kMeta32Bytes = 2 * kP * 16;
static_assert(kMeta32Off % 16 == 0, "float4 metadata rows");
constexpr int kMmaSmem = kMeta32Off + kWarps * kMeta32Bytes + 128;

// 2^x with the SFU (inputs are logit differences <= 0 or -inf)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = a * b: the accumulator input is the constant zero (no registers to clear first)
__device__ __forceinline__ void mma16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
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

// (scale', zero') of both groups of one row from its four compact-format index bytes.
// Byte k of m as an exact float, without an integer conversion: the float 2^23 + byte, minus 2^23.
__device__ __forceinline__ float byte_f(uint32_t m, int k) {
  return __uint_as_float(__byte_perm(m, 0x4B000000u, 0x7540u | (uint32_t)k)) - 8388608.f;
}
__device__ __forceinline__ void u8_row_meta(uint32_t m, const float (&c)[6], float2& g0, float2& g1) {
  // the same values as u8_scale_zero: scale' = (mx8 - mn8) E (an exact difference), zero' = fma(mn8, D, -T)
  const float mn0 = byte_f(m, 0), mx0 = byte_f(m, 1), mn1 = byte_f(m, 2), mx1 = byte_f(m, 3);
  g0 = make_float2(__fmul_rn(mx0 - mn0, c[2]), __fmaf_rn(mn0, c[1], -c[0]));
  g1 = make_float2(__fmul_rn(mx1 - mn1, c[5]), __fmaf_rn(mn1, c[4], -c[3]));
}

// Codebook format: the fp16 value 1024 + k_c of code c from the codebook bytes `lut` (k_0 .. k_3):
// one byte permute per register. sel holds two codes in its bits 0-1 and 8-9 (results in the low and
// the high half); the other selector nibbles pick the constant byte 0x64, fp16 1024's high byte.
__device__ __forceinline__ uint32_t cb_lookup(uint32_t lut, uint32_t sel) {
  return __byte_perm(lut, 0x64646464u, (sel & 0x0303u) | 0x4040u);
}
// The same level as the fp16 subnormal k_c 2^-24 (high bytes zero): the key operand, which then needs no
// constant part cancelled after the tensor cores' truncating accumulation.
__device__ __forceinline__ uint32_t cb_lookup_sub(uint32_t lut, uint32_t sel) {
  return __byte_perm(lut, 0u, (sel & 0x0303u) | 0x4040u);
}

// First page (of n) of split s. Even: floor(s n / nsplit). Folded: the first nsplit - nbf splits take q
// pages each and the last nbf take q - bf_fold (q chosen so the pages add up to n; if n is too short for
// that, the light splits take none), the boundaries rounded down from the exact quotas.
__device__ __forceinline__ int split_start(const FusedArgs& fa, int n, int s) {
  if (fa.bf_fold <= 0) return (int)((long long)s * n / fa.nsplit);
  if (s >= fa.nsplit) return n;
  const int np = fa.nsplit - fa.nbf;                // splits without a BF16 page
  const long long nb = fa.nbf, beta = fa.bf_fold;
  // quotas as fractions over the common denominator: plain q = (n + nb beta) / nsplit, light q - beta;
  // if n < np beta the light splits take nothing and the plain ones n / np
  if ((long long)n >= (long long)np * beta || np == 0) {
    const long long num = (long long)n + nb * beta;  // q = num / nsplit
    if (s <= np) return (int)((long long)s * num / fa.nsplit);
    return (int)(((long long)s * num - (long long)(s - np) * beta * fa.nsplit) / fa.nsplit);
  }
  return s <= np ? (int)((long long)s * n / np) : n;
}

// History split `split` of group (b, h): see the file comment. FMT: the pool's metadata format,
// kFmtF16, kFmtU8 (compact (mn8, mx8) metadata, 4608-byte blocks staged in the same 5120-byte slots) or
// kFmtCB (codebook levels k_c instead of the codes, fp16 range / 255 as the scale).
template <int NT, int FMT>
__device__ __forceinline__ void int2_split(const LayerView& lv, const DecodeWorkspace& ws, const FusedArgs& fa,
                                           uint8_t* smem, int split, int h, int b, unsigned long long* trace) {
  const int* __restrict__ seq_lens = fa.seq_lens;
  const int* __restrict__ hist_pt = fa.hist_pt;
  const int max_hist_pages = fa.max_hist_pages;
  int& any_timeout = *reinterpret_cast<int*>(smem + kWarps * kStages * kBlockBytes + kWarps * kStages * 8);
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int gq = lv.hq / lv.hkv;
  constexpr bool U8 = FMT == kFmtU8, CB = FMT == kFmtCB;
  if (tid == 0) any_timeout = 0;
  __syncthreads();

  // ---- pages of this warp --------------------------------------------------------
  const int L = seq_lens[b] + fa.len_add;
  int Lh = max(0, L - lv.sink - lv.recent);
  int npages = (Lh + kP - 1) / kP;
  if (npages > max_hist_pages) {
    if (tid == 0 && split == 0) flag(lv.status, OSCAR_STATUS_BAD_SEQLEN);
    npages = max_hist_pages;
    Lh = npages * kP;
  }
  // The request's pages from hist_start on are spread over the splits: evenly (split s starts at page
  // hist_start + floor(s n / nsplit), n = npages - hist_start), or, with the BF16 pages folded into the
  // last nbf splits, with those splits bf_fold pages lighter (split_start).
  const int nown = npages - fa.hist_start;
  if (nown < 0 && tid == 0 && split == 0) flag(lv.status, OSCAR_STATUS_BAD_SEQLEN);   // shorter than the shared prefix
  const int p0 = fa.hist_start + split_start(fa, max(nown, 0), split) + w;
  const int p1 = fa.hist_start + split_start(fa, max(nown, 0), split + 1);
  const int my_pages = p0 < p1 ? (p1 - p0 + kWarps - 1) / kWarps : 0;
  const int* pt = hist_pt + (size_t)b * max_hist_pages;

  uint8_t* stage0 = smem + (size_t)w * kStages * kBlockBytes;
  const uint32_t stage_s = smem_addr(stage0);
  const uint32_t bar_s = smem_addr(smem + kWarps * kStages * kBlockBytes) + w * kStages * 8;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(bar_s + 8 * s);
  }
  __syncwarp();

  // issue the load of the warp's i-th page (id pid) into stage i % kStages; returns whether it was issued
  auto issue = [&](int i, int pid) -> bool {
    if (pid < 0 || pid >= lv.n_int2) {
      if (lane == 0) flag(lv.status, OSCAR_STATUS_BAD_PAGE);
      return false;
    }
    if (lane == 0) {
      const int s = i % kStages;
      bulk_load_hint(stage_s + s * kBlockBytes, int2_block(lv, pid, h), U8 ? kBlockBytesU8 : kBlockBytes, bar_s + 8 * s,
                     l2_evict_first());
    }
    return true;
  };
  uint32_t issued = 0;                 // bit s: a load is outstanding in stage s
  // Only the first page of each warp is requested up front: with every warp of
  // the grid asking for one page the first burst lands early, and the later
  // stages are requested once it has (below). Before the programmatic wait only
  // pages the preceding append cannot touch are fetched: it writes one row of
  // the last history page (the demoted token).
  // Page ids are read from the page table a stage ahead of their use.
  int pids[kStages];
#pragma unroll
  for (int k = 0; k < kStages; ++k) pids[k] = k < my_pages ? pt[p0 + kWarps * k] : 0;
  if (my_pages > 0 && p0 < npages - 1 && issue(0, pids[0])) issued |= 1u;
  pdl_wait();
  if (trace != nullptr && tid == 0) trace[7] = global_ns();                  // the programmatic wait returned
  if (my_pages > 0 && p0 >= npages - 1 && issue(0, pids[0])) issued |= 1u;
  auto issue_rest = [&]() {            // pages 1 .. kStages - 1, once page 0 is in (or was never requested)
#pragma unroll
    for (int k = 1; k < kStages; ++k)
      if (k < my_pages && issue(k, pids[k])) issued |= 1u << k;
  };

  // ---- per-lane constants -------------------------------------------------------
  // largest V clip threshold of the head (every warp reduces all 128): it bounds every V scale, hence
  // the P.V weights' range (below)
  float4 tv4 = make_float4(0.f, 0.f, 0.f, 0.f);
  if constexpr (!CB) tv4 = *reinterpret_cast<const float4*>(lv.params + (size_t)h * kParamFloats + kTauVOff + 4 * lane);
  float kmc[6], vmc[6];                // compact format: {T, D, E} of groups 0, 1 for K and for V
  uint32_t klut = 0, vlut = 0;         // codebook format: the bytes k_0 .. k_3 of K and of V
  if constexpr (CB) {
    const float* ck = cb_consts(lv, h, OSCAR_KIND_K);
    const float* cv = cb_consts(lv, h, OSCAR_KIND_V);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      klut |= (uint32_t)ck[i] << (8 * i);
      vlut |= (uint32_t)cv[i] << (8 * i);
    }
  }
  if constexpr (U8) {
    const float* mk = meta_consts(lv, h, OSCAR_KIND_K);
    const float* mv = meta_consts(lv, h, OSCAR_KIND_V);
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      kmc[i] = mk[i];
      kmc[3 + i] = mk[4 + i];
      vmc[i] = mv[i];
      vmc[3 + i] = mv[4 + i];
    }
  }
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
  // the logits' scale and zero-point constants per head (the key operands carry no constant part, so
  // each key tile's accumulator starts from zero)
  // The logit is cF (s0 a0 + s1 a1 + z0 cZ0 / cF + z1 cZ1 / cF): the page keeps the bracket (X), the
  // softmax applies cF (> 0) to its maximum and inside the exponential. Heads past the group: cF = 1, cZ = 0.
  float cF[NT], cZ0[NT], cZ1[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int head = 4 * nt + t;
    cF[nt] = 1.f;
    cZ0[nt] = cZ1[nt] = 0.f;
    if (head < gq) {
      const float* qc = ws.qconst + ((size_t)b * lv.hq + h * gq + head) * kQConst;
      cF[nt] = qc[kQF] * 16777216.f;               // 2^24: the codes (or levels) were fed as subnormals
      cZ0[nt] = __fdiv_rn(qc[kQZ0], cF[nt]);
      cZ1[nt] = __fdiv_rn(qc[kQZ1], cF[nt]);
    }
  }

  // the softmax reference's lag (the codebook format, whose weights' low parts matter, keeps p <= 1)
  constexpr float lag = CB ? 0.f : kLag;
  // P.V weights (non-codebook formats): the V codes are fed like the keys', as fp16 subnormals
  // c 4^pos 2^-24 masked in place, so the weights of the tokens at code position pos carry
  // 4^-pos 2^sw. With s < 2^e (s <= fp16(2 tau_max / 3), tau_max < 2^e) and p < 2^kLag (the softmax
  // below), sw = 15 - e - kLag keeps every weight below 2^15; the accumulators then hold
  // sum p s c 2^(sw - 24).
  float wsc = 1.f, wback = 1.f;
  if constexpr (!CB) {
    float tv = fmaxf(fmaxf(fabsf(tv4.x), fabsf(tv4.y)), fmaxf(fabsf(tv4.z), fabsf(tv4.w)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tv = fmaxf(tv, __shfl_xor_sync(0xffffffffu, tv, o));
    int sw = 0;
    if (tv > 0.f && tv < INFINITY) {
      int e;
      frexpf(tv, &e);                              // tv = m 2^e, 0.5 <= m < 1
      sw = min(max(15 - e - (int)lag, -60), 60);
    }
    wsc = exp2f((float)sw);
    wback = exp2f((float)(24 - sw));
  }
  // this lane converts metadata rows lane and lane + 32 of each page: their V scales carry the weight
  // factor of their code position 2 ((row >> 4) & 1) + ((row >> 3) & 1) (the same for both rows;
  // codebook: 256 / 255 instead), their K scales 1 / 255 in the codebook format
  const int vpos = 2 * ((lane >> 4) & 1) + ((lane >> 3) & 1);
  const float vfac = CB ? 256.f / 255.f : wsc * exp2f(-2.f * (float)vpos);
  const float kfac = CB ? 1.f / 255.f : 1.f;
  float4* meta_w = reinterpret_cast<float4*>(smem + kMeta32Off + w * kMeta32Bytes);   // [K, V][64 rows]

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

  for (int i = 0, s = 0; i < my_pages; ++i, s = (s + 1 == kStages) ? 0 : s + 1) {   // s = i % kStages
    const int pid_ahead = (i + kStages < my_pages) ? pt[p0 + kWarps * (i + kStages)] : 0;   // used after this page
    if (issued & (1u << s)) {
      const bool landed = __all_sync(0xffffffffu, mbar_wait(bar_s + 8 * s, (phase >> s) & 1u));
      if (trace != nullptr && i == 0 && tid == 0) trace[3] = global_ns();      // first page of warp 0 landed
      if (!landed) {                   // warp-uniform decision: the shuffles and MMAs below need every lane
        timed_out = true;
        break;
      }
      phase ^= 1u << s;
      issued &= ~(1u << s);
      if (i == 0) issue_rest();
      const uint8_t* blk = stage0 + s * kBlockBytes;
      const int ntok = min(kP, Lh - (p0 + kWarps * i) * kP);

      // ---- the page's metadata as float32 rows, converted once for the warp (rows past the end zero) ----
#pragma unroll
      for (int kind = 0; kind < 2; ++kind) {
        float4 m[2];                               // rows lane, lane + 32
        if constexpr (U8) {
          const uint8_t* mb = blk + (kind ? kVMetaOffU8 : kKMetaOff);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            float2 g0, g1;
            u8_row_meta(*reinterpret_cast<const uint32_t*>(mb + 4 * (lane + 32 * r)), kind ? vmc : kmc, g0, g1);
            m[r] = make_float4(g0.x, g0.y, g1.x, g1.y);
          }
        } else {
          const uint8_t* mb = blk + (kind ? kVMetaOff : kKMetaOff);
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const uint2 u = *reinterpret_cast<const uint2*>(mb + 8 * (lane + 32 * r));
            const float2 a0 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
            const float2 a1 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
            m[r] = make_float4(a0.x, a0.y, a1.x, a1.y);
          }
        }
        const float f = kind ? vfac : kfac;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if (kind == 1 || CB) {
            m[r].x = __fmul_rn(m[r].x, f);
            m[r].z = __fmul_rn(m[r].z, f);
          }
        }
        if (ntok < kP) {
#pragma unroll
          for (int r = 0; r < 2; ++r)
            if (lane + 32 * r >= ntok) m[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        meta_w[kind * kP + lane] = m[0];
        meta_w[kind * kP + lane + 32] = m[1];
      }
      __syncwarp();

      // ---- logits of the page's 64 tokens -----------------------------------------
      float lg[4][NT][2];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int r0 = 16 * mt + g, r1 = r0 + 8;
        // words t (channels 16t .. 16t+15, group 0) and t + 4 (group 1) of rows r0, r1
        const uint32_t kx[2] = {*reinterpret_cast<const uint32_t*>(blk + kKCodesOff + r0 * 32 + 4 * t),
                                *reinterpret_cast<const uint32_t*>(blk + kKCodesOff + r0 * 32 + 16 + 4 * t)};
        const uint32_t ky[2] = {*reinterpret_cast<const uint32_t*>(blk + kKCodesOff + r1 * 32 + 4 * t),
                                *reinterpret_cast<const uint32_t*>(blk + kKCodesOff + r1 * 32 + 16 + 4 * t)};
        float c[2][NT][4];                         // per group; starts from -offset: the MMAs add the biased sums
#pragma unroll
        for (int G = 0; G < 2; ++G) {
          // codes 0-3 of each 16-bit half from the word, codes 4-7 from the word shifted right by 8
          const uint32_t wx[2] = {kx[G], kx[G] >> 8};
          const uint32_t wy[2] = {ky[G], ky[G] >> 8};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t a0, a1, a2, a3;
            if constexpr (CB) {
              // k rows (2t, 2t+1): channels (16t + j, 16t + 4 + j) of the word (bytes 0, 1 at bits 2j);
              // (2t+8, 2t+9): channels (16t + 8 + j, 16t + 12 + j) (bytes 2, 3)
              a0 = cb_lookup_sub(klut, kx[G] >> (2 * j));
              a1 = cb_lookup_sub(klut, ky[G] >> (2 * j));
              a2 = cb_lookup_sub(klut, kx[G] >> (2 * j + 16));
              a3 = cb_lookup_sub(klut, ky[G] >> (2 * j + 16));
            } else {
              // the masked bits as fp16 subnormals c 4^(p mod 4) 2^-24, p the code's position (no bias, no
              // conversion; the query fragments carry 4^-(p mod 4))
              const uint32_t m0 = 0x00030003u << (4 * (j & 1)), m1 = 0x000C000Cu << (4 * (j & 1));
              a0 = wx[j >> 1] & m0;                    // row r0, codes 2j (k rows 2t, 2t+1)
              a1 = wy[j >> 1] & m0;                    // row r1
              a2 = wx[j >> 1] & m1;                    // row r0, codes 2j+1 (k rows 2t+8, 2t+9)
              a3 = wy[j >> 1] & m1;                    // row r1
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              if (j == 0) mma16816_z(c[G][nt], a0, a1, a2, a3, qf[4 * G + j][nt][0], qf[4 * G + j][nt][1]);
              else mma16816(c[G][nt], a0, a1, a2, a3, qf[4 * G + j][nt][0], qf[4 * G + j][nt][1]);
            }
          }
        }
        // (scale, zero of group 0, scale, zero of group 1) of rows r0, r1 (codebook: scale = range / 255, the
        // dequantised value being zero + scale k_c)
        const float4 k0 = meta_w[r0], k1 = meta_w[r1];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float a00 = c[0][nt][0] + c[0][nt][1], a01 = c[1][nt][0] + c[1][nt][1];   // row r0: hi + lo per group
          const float a10 = c[0][nt][2] + c[0][nt][3], a11 = c[1][nt][2] + c[1][nt][3];   // row r1
          lg[mt][nt][0] = fmaf(k0.x, a00, fmaf(k0.z, a01, fmaf(k0.y, cZ0[nt], k0.w * cZ1[nt])));
          lg[mt][nt][1] = fmaf(k1.x, a10, fmaf(k1.z, a11, fmaf(k1.y, cZ0[nt], k1.w * cZ1[nt])));
        }
        if (ntok < kP) {                           // ragged last page: rows past the end take no weight
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (r0 >= ntok) lg[mt][nt][0] = -INFINITY;
            if (r1 >= ntok) lg[mt][nt][1] = -INFINITY;
          }
        }
      }

      // ---- online softmax with a lagging reference -------------------------------------
      // The weights 2^(logit - mrun) use the running reference mrun of their head. Only if a logit of the
      // page exceeds it by more than kLag (the first page always does) is the reference raised to the
      // page's maximum, the state rescaled and the weights' exponents taken again: the common path
      // needs one vote, not the maximum's shuffles, before its exponentials. Weights stay below 2^kLag.
      float pw[4][NT][2];                          // log2 of the weights
      bool raise = false;
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            pw[mt][nt][r] = fmaf(cF[nt], lg[mt][nt][r], -mrun[nt]);
            raise |= pw[mt][nt][r] > lag;          // +inf against a reference of -inf
          }
      if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float mx = -INFINITY;
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) mx = fmaxf(mx, fmaxf(lg[mt][nt][0], lg[mt][nt][1]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mnew = fmaxf(mrun[nt], cF[nt] * mx);
          const float al = (mnew > mrun[nt]) ? exp2f(mrun[nt] - mnew) : 1.f;
          lsum[nt] *= al;
          zacc[nt][0] *= al;
          zacc[nt][1] *= al;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][mt][e] *= al;
          mrun[nt] = mnew;
#pragma unroll
          for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r) pw[mt][nt][r] = fmaf(cF[nt], lg[mt][nt][r], -mrun[nt]);
        }
      }

      // ---- P.Vhat over the page's four 16-token tiles -----------------------------------
      // weights p * scale of the page's 64 tokens: the B fragments of the four 16-token tiles; the codebook
      // format also keeps their fp16 rounding remainders (a second MMA per tile: its levels span the whole
      // range, so the weights' rounding would otherwise dominate its error)
      uint32_t bf[4][NT][2];
      uint32_t bfl[CB ? 4 : 1][NT][2];
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        const int r0 = 16 * kt + g, r1 = r0 + 8;
        // (scale x weight factor, zero) of groups 0, 1 of rows r0, r1 (codebook: range x 256 / 255, the V
        // operand holding k_c / 256); zero rows past the end
        const float4 v0 = meta_w[kP + r0], v1 = meta_w[kP + r1];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float pa = fast_exp2(pw[kt][nt][0]);
          const float pb = fast_exp2(pw[kt][nt][1]);
          lsum[nt] += pa + pb;
          zacc[nt][0] = fmaf(pa, v0.y, fmaf(pb, v1.y, zacc[nt][0]));
          zacc[nt][1] = fmaf(pa, v0.w, fmaf(pb, v1.w, zacc[nt][1]));
          // lane (g, t): the weights of token row g (rows 0-7) and g + 8 of the tile for head t, groups 0 and 1;
          // the transposes give lane (g', t') B rows k = (2t', 2t'+1) and (2t'+8, 2t'+9) of column g'
          const float x0 = pa * v0.x, x1 = pa * v0.z, x2 = pb * v1.x, x3 = pb * v1.z;
          const uint32_t h01 = pack_f16x2(x0, x1), h23 = pack_f16x2(x2, x3);
          bf[kt][nt][0] = movmatrix_t(h01);
          bf[kt][nt][1] = movmatrix_t(h23);
          if constexpr (CB) {
            const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
            const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
            bfl[kt][nt][0] = movmatrix_t(pack_f16x2(x0 - f01.x, x1 - f01.y));
            bfl[kt][nt][1] = movmatrix_t(pack_f16x2(x2 - f23.x, x3 - f23.y));
          }
        }
      }
      // P.Vhat: tile mt takes channels 16 g + mt (rows g) and 16 g + 8 + mt (rows g + 8). Word t of a
      // channel's V codes holds exactly this lane's k pairs of the page: (2t, 2t+1) = tokens (16 kt + 2t, + 1)
      // at code position 2 kt, (2t+8, 2t+9) = tokens (16 kt + 2t + 8, + 9) at position 2 kt + 1
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const uint32_t wa = *reinterpret_cast<const uint32_t*>(blk + v_chan_off(16 * g + mt) + 4 * t);
        const uint32_t wb = *reinterpret_cast<const uint32_t*>(blk + v_chan_off(16 * g + 8 + mt) + 4 * t);
        const uint32_t xa[2] = {wa, wa >> 8}, xb[2] = {wb, wb >> 8};   // positions 0-3, then 4-7 at 0-3
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
          const int pp = (2 * kt) & 3, hh = kt >> 1;          // positions 2 kt, 2 kt + 1 of half-word hh
          uint32_t a0, a1, a2, a3;
          if constexpr (CB) {
            // level k_c / 256 exactly: the two codes (bits 2p and 16 + 2p) gathered 8 bits apart as the lookup's
            // selector wants them
            auto sel = [](uint32_t x, int p) { return ((x >> (2 * p)) & 3u) | ((x >> (8 + 2 * p)) & 0x300u); };
            a0 = exact_codes(cb_lookup(vlut, sel(xa[hh], pp)), 4);
            a1 = exact_codes(cb_lookup(vlut, sel(xb[hh], pp)), 4);
            a2 = exact_codes(cb_lookup(vlut, sel(xa[hh], pp + 1)), 4);
            a3 = exact_codes(cb_lookup(vlut, sel(xb[hh], pp + 1)), 4);
          } else {
            // the masked bits as fp16 subnormals c 4^p 2^-24 (the weights carry 4^-p)
            a0 = xa[hh] & (0x00030003u << (2 * pp));
            a1 = xb[hh] & (0x00030003u << (2 * pp));
            a2 = xa[hh] & (0x00030003u << (2 * pp + 2));
            a3 = xb[hh] & (0x00030003u << (2 * pp + 2));
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816(acc[nt][mt], a0, a1, a2, a3, bf[kt][nt][0], bf[kt][nt][1]);
            if constexpr (CB) mma16816(acc[nt][mt], a0, a1, a2, a3, bfl[kt][nt][0], bfl[kt][nt][1]);
          }
        }
      }
    } else if (i == 0) {
      issue_rest();                    // page 0 was not requested (bad page id): the rest still is
    }
    __syncwarp();
    const int next = i + kStages;
    if (next < my_pages && issue(next, pid_ahead)) issued |= 1u << s;
  }

  if (timed_out) {
    // give the copies still in flight a bounded chance to land before the buffers are reused
    if (lane == 0) flag(lv.status, OSCAR_STATUS_TIMEOUT);
    for (int s = 0; s < kStages; ++s)
      if (issued & (1u << s)) mbar_wait(bar_s + 8 * s, (phase >> s) & 1u);
    any_timeout = 1;
  }

  if (trace != nullptr && lane == 0) atomicMax(&trace[4], global_ns());      // last warp's main loop done
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
  // rows of 132 floats: the four 16-byte stores of the 8 lanes of a quarter warp hit distinct banks
  constexpr int kCaStride = kD + 4;
  float* cm = reinterpret_cast<float*>(smem);     // [kWarps][8] running max
  float* cl = cm + kWarps * 8;                    // [kWarps][8] running sum
  float* ca = cl + kWarps * 8;                    // [kWarps][8][kCaStride] accumulators
  const int grp = g >> 2;                         // channels 16g .. 16g+15 lie in group g / 4
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int head = 4 * nt + t;
    if (g == 0) {
      cm[w * 8 + head] = mrun[nt];
      cl[w * 8 + head] = lsum[nt];
    }
    const float zs = grp ? zacc[nt][1] : zacc[nt][0];
    float v[16];                                  // channels 16g .. 16g + 15
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      // the accumulators hold sum p s c 2^(sw - 24) (the codebook build: exactly scaled, its levels fed / 256
      // and its P operand carrying the 256): scale back, add the zero-point part
      v[mt] = fmaf(grp ? acc[nt][mt][1] : acc[nt][mt][0], wback, zs);
      v[8 + mt] = fmaf(grp ? acc[nt][mt][3] : acc[nt][mt][2], wback, zs);
    }
    float4* dst = reinterpret_cast<float4*>(ca + (w * 8 + head) * kCaStride + 16 * g);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
  __syncthreads();
  // the query heads unrolled (gq <= 4 NT), so that their shared-memory loads and exponentials overlap
  const bool ok = !any_timeout;
#pragma unroll
  for (int hh = 0; hh < 4 * NT; ++hh) {
    if (hh >= gq) break;
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, cm[ww * 8 + hh]);
    float Ls = 0.f, A = 0.f;
    if (M != -INFINITY && ok) {
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) {
        const float f = fast_exp2(cm[ww * 8 + hh] - M);    // 0 for a warp without pages (m = -inf)
        Ls = fmaf(cl[ww * 8 + hh], f, Ls);
        A = fmaf(ca[(ww * 8 + hh) * kCaStride + tid], f, A);
      }
    } else {
      M = -INFINITY;
    }
    float* part = part_row(ws, b, lv.hq, h * gq + hh, split);
    if (tid == 0) {
      part[0] = M;
      part[1] = Ls;
    }
    part[4 + tid] = A;
  }
}

// grid = (nsplit + nbf, hkv, B), block = 128: history splits, then one CTA per BF16 page.
// MINB resident CTAs per SM (the register budget): 3 for grids of one or two waves (more registers, more
// independent work per warp), 4 for grids of many waves (more warps to hide latency).
template <int NT, int MINB, int FMT>
__global__ void __launch_bounds__(128, MINB) k_decode_mma(LayerView lv, DecodeWorkspace ws, FusedArgs fa) {
  TimelineSpan timeline_span(lv, kTlDecodeMma);
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
  const int h = blockIdx.y, b = blockIdx.z;
  // optional timeline record of this CTA (ns, %globaltimer):
  // [0] linear CTA id, [1] SM id, [2] start, [3] first history page landed (warp 0),
  // [4] last warp's main loop done, [5] partials written, [6] 0, [7] the programmatic wait returned
  // (history CTAs)
  const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  unsigned long long* trace =
      (ws.cta_trace != nullptr && (int)cta < ws.trace_cap) ? ws.cta_trace + 8ull * cta : nullptr;
  if (trace != nullptr) {
    if (threadIdx.x == 0) {
      trace[0] = cta;
      trace[1] = sm_id();
      trace[2] = global_ns();
      trace[3] = trace[4] = trace[5] = trace[6] = trace[7] = 0;
    }
    __syncthreads();
  }
  pdl_launch_dependents();                         // the merge kernel may be scheduled now; it waits for this grid
  if (blockIdx.x < fa.nsplit) {
    if (fa.bf_fold > 0 && (int)blockIdx.x >= fa.nsplit - fa.nbf && threadIdx.x == 0) {
      // this split's BF16 page, read after its history pages: into L2 now (a hint; the append may still
      // write one row of it, which L2 then holds)
      const int c = (int)blockIdx.x - (fa.nsplit - fa.nbf);
      const int page = fa.bf16_pt[(size_t)b * ((lv.sink + lv.recent) / kP) + c];
      if (page >= 0 && page < lv.n_bf16)
        l2_prefetch(lv.bf16 + ((size_t)page * lv.hkv + h) * kBf16BlockBytes, kBf16BlockBytes, l2_evict_last());
    }
    int2_split<NT, FMT>(lv, ws, fa, smem, blockIdx.x, h, b, trace);
    // this split's BF16 page, in the ring's memory (its index recomputed here: nothing stays live across
    // the history loop)
    if (fa.bf_fold > 0 && (int)blockIdx.x >= fa.nsplit - fa.nbf) {
      __syncthreads();
      bf16_page(lv, ws, fa, smem, (int)blockIdx.x - (fa.nsplit - fa.nbf), blockIdx.y, blockIdx.z);
    }
  } else {
    bf16_page(lv, ws, fa, smem, blockIdx.x - fa.nsplit, h, b);
  }
  if (trace != nullptr && threadIdx.x == 0) trace[5] = global_ns();
}

}  // namespace

// the kernel build for the layout's metadata format, the GQA width and the occupancy the split policy chose
template <int FMT>
static cudaError_t launch_fmt(cudaLaunchConfig_t& cfg, const LayerView& lv, const DecodeWorkspace& ws,
                              const FusedArgs& fa, int occupancy) {
  if (lv.hq / lv.hkv > 4) return cudaLaunchKernelEx(&cfg, k_decode_mma<2, 2, FMT>, lv, ws, fa);
  if (occupancy == 4) return cudaLaunchKernelEx(&cfg, k_decode_mma<1, 4, FMT>, lv, ws, fa);
  return cudaLaunchKernelEx(&cfg, k_decode_mma<1, 3, FMT>, lv, ws, fa);
}

int launch_decode_mma(const LayerView& lv, const DecodeWorkspace& ws, const DecodeArgs& a, float scale_log2,
                      cudaStream_t st) {
  FusedArgs fa = {};
  fa.seq_lens = a.seq_lens;
  fa.len_add = a.len_add;
  fa.hist_pt = a.hist_pt;
  fa.max_hist_pages = a.max_hist_pages;
  fa.nsplit = a.nsplit;
  fa.nbf = a.nbf;
  fa.bf_fold = a.nsplit >= a.nbf ? kBf16FoldPages : 0;
  fa.hist_start = a.shared_pages;
  fa.bf_slot0 = a.nsplit + a.nsplit_shared;
  fa.bf16_pt = a.bf16_pt;
  fa.q = static_cast<const __nv_bfloat16*>(a.q);
  fa.scale_log2 = scale_log2;
  fa.out = a.out;
  fa.out_dtype = a.out_dtype;
  fa.lse = a.lse;
  // programmatic dependent of the query prologue: starts early, prefetches, then waits
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(a.nsplit + (fa.bf_fold > 0 ? 0 : a.nbf), lv.hkv, a.B);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = kMmaSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  // right behind a profiling event the launch is ordered after the prologue anyway: without the attribute
  // (which lets it start early only behind a kernel)
  cfg.numAttrs = (a.ev0 != nullptr && a.nsplit_shared == 0) ? 0 : 1;
  cudaError_t e;
  if (lv.meta_u8) e = launch_fmt<kFmtU8>(cfg, lv, ws, fa, a.mma_occupancy);
  else if (lv.meta_cb) e = launch_fmt<kFmtCB>(cfg, lv, ws, fa, a.mma_occupancy);
  else e = launch_fmt<kFmtF16>(cfg, lv, ws, fa, a.mma_occupancy);
  return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int configure_mma_kernels() {
  const void* fns[9] = {reinterpret_cast<const void*>(k_decode_mma<1, 3, kFmtF16>),
                        reinterpret_cast<const void*>(k_decode_mma<1, 4, kFmtF16>),
                        reinterpret_cast<const void*>(k_decode_mma<2, 2, kFmtF16>),
                        reinterpret_cast<const void*>(k_decode_mma<1, 3, kFmtU8>),
                        reinterpret_cast<const void*>(k_decode_mma<1, 4, kFmtU8>),
                        reinterpret_cast<const void*>(k_decode_mma<2, 2, kFmtU8>),
                        reinterpret_cast<const void*>(k_decode_mma<1, 3, kFmtCB>),
                        reinterpret_cast<const void*>(k_decode_mma<1, 4, kFmtCB>),
                        reinterpret_cast<const void*>(k_decode_mma<2, 2, kFmtCB>)};
  for (const void* f : fns) {
    if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmem) != cudaSuccess)
      return OSCAR_ERR_CUDA;
    if (set_max_shared_carveout(f) != OSCAR_OK) return OSCAR_ERR_CUDA;
  }
  return OSCAR_OK;
}

}  // namespace oscar
