// Decode attention over the mixed-precision pool, CUDA-core path, and the
// pieces every decode path shares: the query prologue, the BF16 segment
// kernel and the all-BF16 comparison kernel (sm_103a). The log-sum-exp merge
// is in merge.cu.
//
// News article "超越 TurboQuant…OSCAR…", section "OSCAR 的设计思路": the INT2
// kernel unpacks, restores scale/zero and accumulates in floating point; the
// BF16 kernel handles sink and recent; an online-softmax merge combines them.
// MarkTechPost article "Together AI 开源 OSCAR…", section "服务系统：混合精度缓存
// 布局": the read path undoes the rotation; with R_V absorbed into the
// projections no value inverse rotation is needed. Here the key side is
// handled by rotating the query once (q R_K), which equals inverse-rotating
// every dequantised key because R_K is orthogonal.
//
// Softmax bookkeeping is in base 2: logits are scaled by sm_scale*log2(e),
// partials hold (m, l, acc) with l = sum 2^(logit - m), acc = sum 2^(logit - m) v.
#include "kernels.cuh"
#include "rotate.cuh"
#include "tma.cuh"
#include "timeline.cuh"

namespace oscar {

namespace {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, s));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) v += __shfl_xor_sync(0xffffffffu, v, s);
  return v;
}

__device__ __forceinline__ float* part_ptr(float* partials, int b, int hq_total, int hq, int nslots, int s) {
  return partials + (((size_t)b * hq_total + hq) * nslots + s) * kPartFloats;
}

// Online-softmax state of GQ heads over one chunk of up to 64 tokens whose
// logits (base 2) sit in pbuf[GQ][64]; -inf marks an absent token. Converts
// pbuf to probabilities relative to the new running max and records the
// rescale factor of the previous accumulators in alpha. 128 threads.
template <int GQ>
__device__ __forceinline__ void softmax_chunk(float (&pbuf)[GQ][kP], float* mrow, float* lrow, float* alpha) {
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int hh = wib; hh < GQ; hh += 4) {
    const float l0 = pbuf[hh][lane], l1 = pbuf[hh][lane + 32];
    const float cm = warp_max(fmaxf(l0, l1));
    const float m_old = mrow[hh];
    const float m_new = fmaxf(m_old, cm);
    float p0 = 0.f, p1 = 0.f, al = 1.f;
    if (m_new != -INFINITY) {
      p0 = exp2f(l0 - m_new);
      p1 = exp2f(l1 - m_new);
      al = exp2f(m_old - m_new);
    }
    const float ps = warp_sum(p0 + p1);
    pbuf[hh][lane] = p0;
    pbuf[hh][lane + 32] = p1;
    if (lane == 0) {
      alpha[hh] = al;
      lrow[hh] = lrow[hh] * al + ps;
      mrow[hh] = m_new;
    }
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// INT2 history, CUDA cores. grid = (nsplit, hkv, B), block = 128.
// A CTA walks its range of history pages; per 64-token page it computes the
// logits of all GQ heads (thread per (token, head)), updates the online
// softmax, then accumulates P.Vhat (thread per rotated channel).
template <int GQ, bool CB>
__global__ void __launch_bounds__(128) k_int2_simt(LayerView lv, DecodeWorkspace ws, const int* __restrict__ seq_lens,
                                                   const int* __restrict__ hist_pt, int max_hist_pages,
                                                   int pages_per_split, float scale_log2, int len_add) {
  TimelineSpan timeline_span(lv, kTlInt2Simt);
  __shared__ __align__(16) uint8_t blk[kBlockBytes];
  __shared__ float2 msz[2][kP][kNG];     // [K, V][token][group] (scale', zero') of the staged page
  __shared__ float mcs[32];              // compact format {T, D, E, 0} per (kind, group); codebook per kind
  __shared__ float qs[GQ][kD];
  __shared__ float qg[GQ][kNG];
  __shared__ float pbuf[GQ][kP];
  __shared__ float mrow[GQ], lrow[GQ], alpha[GQ];
  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int hq0 = h * GQ;
  const int L = seq_lens[b] + len_add;
  int Lh = max(0, L - lv.sink - lv.recent);
  int npages = (Lh + kP - 1) / kP;
  if (npages > max_hist_pages) {
    if (tid == 0 && s == 0) flag(lv.status, OSCAR_STATUS_BAD_SEQLEN);
    npages = max_hist_pages;
    Lh = npages * kP;
  }
  const int p0 = s * pages_per_split, p1 = min(p0 + pages_per_split, npages);
  for (int i = tid; i < GQ * kD; i += 128) qs[i / kD][i % kD] = ws.qrot[((size_t)b * lv.hq + hq0) * kD + i];
  if (tid < GQ * kNG) qg[tid / kNG][tid % kNG] = ws.qconst[((size_t)b * lv.hq + hq0 + tid / kNG) * kQConst + kQSum0 + tid % kNG];
  if (tid < GQ) { mrow[tid] = -INFINITY; lrow[tid] = 0.f; }
  if (tid < 32) mcs[tid] = lv.params[(size_t)h * kParamFloats + kMetaCOff + tid];
  const float* lvk = mcs + 16;            // codebook levels k_0..k_3 of K (then thresholds), V at + 8
  float acc[GQ];
#pragma unroll
  for (int i = 0; i < GQ; ++i) acc[i] = 0.f;
  __syncthreads();
  for (int page = p0; page < p1; ++page) {
    const int pid = hist_pt[(size_t)b * max_hist_pages + page];
    if (pid < 0 || pid >= lv.n_int2) {
      if (tid == 0) flag(lv.status, OSCAR_STATUS_BAD_PAGE);
      continue;
    }
    const int ntok = min(kP, Lh - page * kP);
    const uint4* src = reinterpret_cast<const uint4*>(int2_block(lv, pid, h));
    uint4* dst = reinterpret_cast<uint4*>(blk);
    for (int i = tid; i < lv.blk_bytes / 16; i += 128) dst[i] = src[i];
    __syncthreads();
    for (int i = tid; i < 2 * kP * kNG; i += 128) {     // metadata of both kinds as float pairs
      const int kind = i / (kP * kNG), tk = (i / kNG) % kP, g = i % kNG;
      float2 sz;
      if (!lv.meta_u8) {
        const __half* m = reinterpret_cast<const __half*>(blk + (kind ? kVMetaOff : kKMetaOff) + tk * kNG * 4) + 2 * g;
        sz = make_float2(__half2float(m[0]), __half2float(m[1]));
        if (CB) sz.x = __fmul_rn(sz.x, 1.f / 255.f);     // range / 255: the dequantised value is zero + that * k
      } else {
        const uint8_t* m = blk + (kind ? kVMetaOffU8 : kKMetaOff) + tk * kNG * 2 + 2 * g;
        const float* c = mcs + 8 * kind + 4 * g;
        sz = u8_scale_zero(m[0], m[1], c[0], c[1], c[2]);
      }
      msz[kind][tk][g] = sz;
    }
    __syncthreads();
    for (int item = tid; item < GQ * kP; item += 128) {
      const int tk = item % kP, hh = item / kP;
      float l = -INFINITY;
      if (tk < ntok) {
        const uint32_t* kw = reinterpret_cast<const uint32_t*>(blk + kKCodesOff + tk * (kD / 4));
        float dot = 0.f;
#pragma unroll
        for (int g = 0; g < kNG; ++g) {
          float a = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint32_t word = kw[g * 4 + w];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const unsigned c = (word >> (2 * i)) & 3u;
              a = fmaf(CB ? lvk[c] : (float)c, qs[hh][g * 64 + w * 16 + i], a);
            }
          }
          dot = fmaf(msz[0][tk][g].x, a, dot);
          dot = fmaf(msz[0][tk][g].y, qg[hh][g], dot);
        }
        l = dot * scale_log2;
      }
      pbuf[hh][tk] = l;
    }
    __syncthreads();
    softmax_chunk<GQ>(pbuf, mrow, lrow, alpha);
    __syncthreads();
    {
      const int c = tid, g = c / kG;
      const int woff = v_chan_off(c);                     // channel-major V codes
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) acc[hh] *= alpha[hh];
      for (int tk = 0; tk < ntok; ++tk) {
        const uint32_t word = *reinterpret_cast<const uint32_t*>(blk + woff + 4 * v_word(tk));
        const unsigned ci = (word >> v_bit(tk)) & 3u;
        const float code = CB ? lvk[8 + ci] : (float)ci;
        const float vhat = fmaf(msz[1][tk][g].x, code, msz[1][tk][g].y);
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) acc[hh] = fmaf(pbuf[hh][tk], vhat, acc[hh]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int hh = 0; hh < GQ; ++hh) {
    float* part = part_ptr(ws.partials, b, lv.hq, hq0 + hh, ws.nslots, s);
    if (tid == 0) { part[0] = mrow[hh]; part[1] = lrow[hh]; }
    part[4 + tid] = acc[hh];
  }
}

// ---------------------------------------------------------------------------
// Attention of GQ query heads (raw q, float in qs) over a list of BF16 tokens,
// in chunks of 64; `locate(i, page, row)` maps list index i to its page block
// and row and returns false for an invalid entry. Leaves (m, l) in mrow/lrow
// and the accumulators of channel threadIdx.x in acc. 128 threads.
template <int GQ, typename Locate>
__device__ __forceinline__ void attend_bf16_list(const uint8_t* __restrict__ pages, int hkv, int h, int n,
                                                 float scale_log2, const Locate& locate,
                                                 __nv_bfloat16 (&ks)[kP][kD + 8], __nv_bfloat16 (&vs)[kP][kD],
                                                 float (&qs)[GQ][kD], float (&pbuf)[GQ][kP], float* mrow,
                                                 float* lrow, float* alpha, int* valid, float (&acc)[GQ]) {
  const int tid = threadIdx.x, wib = tid >> 5, lane = tid & 31;
  for (int c0 = 0; c0 < n; c0 += kP) {
    const int ntok = min(kP, n - c0);
    for (int tk = wib; tk < ntok; tk += 4) {
      int page, row;
      const bool ok = locate(c0 + tk, page, row);
      if (lane == 0) valid[tk] = ok;
      if (ok) {
        const uint8_t* blkp = pages + ((size_t)page * hkv + h) * kBf16BlockBytes;
        const uint2* ksrc = reinterpret_cast<const uint2*>(blkp + (size_t)row * kD * 2);
        const uint2* vsrc = reinterpret_cast<const uint2*>(blkp + (size_t)(kP + row) * kD * 2);
        reinterpret_cast<uint2*>(&ks[tk][0])[lane] = ksrc[lane];
        reinterpret_cast<uint2*>(&vs[tk][0])[lane] = vsrc[lane];
      }
    }
    __syncthreads();
    for (int item = tid; item < GQ * kP; item += 128) {
      const int tk = item % kP, hh = item / kP;
      float l = -INFINITY;
      if (tk < ntok && valid[tk]) {
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < kD / 8; ++i) {
          const uint4 kv = *reinterpret_cast<const uint4*>(&ks[tk][8 * i]);
          const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kv);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 kf = __bfloat1622float2(k2[e]);
            dot = fmaf(kf.x, qs[hh][8 * i + 2 * e], dot);
            dot = fmaf(kf.y, qs[hh][8 * i + 2 * e + 1], dot);
          }
        }
        l = dot * scale_log2;
      }
      pbuf[hh][tk] = l;
    }
    __syncthreads();
    softmax_chunk<GQ>(pbuf, mrow, lrow, alpha);
    __syncthreads();
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) acc[hh] *= alpha[hh];
    for (int tk = 0; tk < ntok; ++tk) {
      if (!valid[tk]) continue;
      const float vv = __bfloat162float(vs[tk][tid]);
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) acc[hh] = fmaf(pbuf[hh][tk], vv, acc[hh]);
    }
    __syncthreads();
  }
}

// BF16 sink + recent segment of the mixed-precision pool. grid = (hkv, B), block = 128.
// Writes its partial into slot `slot` (right after the history splits).
template <int GQ>
__global__ void __launch_bounds__(128) k_bf16_seg(LayerView lv, DecodeWorkspace ws, const __nv_bfloat16* __restrict__ q,
                                                  const int* __restrict__ seq_lens, const int* __restrict__ bf16_pt,
                                                  float scale_log2, int slot, int len_add) {
  TimelineSpan timeline_span(lv, kTlBf16Seg);
  __shared__ __align__(16) __nv_bfloat16 ks[kP][kD + 8];
  __shared__ __align__(16) __nv_bfloat16 vs[kP][kD];
  __shared__ float qs[GQ][kD];
  __shared__ float pbuf[GQ][kP];
  __shared__ float mrow[GQ], lrow[GQ], alpha[GQ];
  __shared__ int valid[kP];
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int hq0 = h * GQ;
  const int L = seq_lens[b] + len_add;
  if (L < 1 && tid == 0) flag(lv.status, OSCAR_STATUS_BAD_SEQLEN);
  const int n_sink = max(0, min(L, lv.sink));
  const int n_rec = L > lv.sink ? min(L - lv.sink, lv.recent) : 0;
  const int bf16_per_req = (lv.sink + lv.recent) / kP;
  for (int i = tid; i < GQ * kD; i += 128) qs[i / kD][i % kD] = __bfloat162float(q[((size_t)b * lv.hq + hq0) * kD + i]);
  if (tid < GQ) { mrow[tid] = -INFINITY; lrow[tid] = 0.f; }
  float acc[GQ];
#pragma unroll
  for (int i = 0; i < GQ; ++i) acc[i] = 0.f;
  __syncthreads();
  const int* pt = bf16_pt + (size_t)b * bf16_per_req;
  const int sink = lv.sink, recent = lv.recent, nb = lv.n_bf16;
  int* status = lv.status;
  auto locate = [&](int i, int& page, int& row) -> bool {
    int pos = i < n_sink ? i : (L - n_rec) + (i - n_sink);
    if (pos < sink) { page = pt[pos / kP]; row = pos % kP; }
    else { const int slot = (pos - sink) % recent; page = pt[sink / kP + slot / kP]; row = slot % kP; }
    if (page < 0 || page >= nb) { flag(status, OSCAR_STATUS_BAD_PAGE); return false; }
    return true;
  };
  attend_bf16_list<GQ>(lv.bf16, lv.hkv, h, n_sink + n_rec, scale_log2, locate, ks, vs, qs, pbuf, mrow, lrow, alpha,
                       valid, acc);
#pragma unroll
  for (int hh = 0; hh < GQ; ++hh) {
    float* part = part_ptr(ws.partials, b, lv.hq, hq0 + hh, ws.nslots, slot);
    if (tid == 0) { part[0] = mrow[hh]; part[1] = lrow[hh]; }
    part[4 + tid] = acc[hh];
  }
}

// ---------------------------------------------------------------------------
// Log-sum-exp merge of the history splits (slots [0, nsplit)) and the BF16
// partial (slot nsplit). grid = (hkv, B), block = 128 (thread = output
// channel). In explicit-V mode the combined history accumulator, which lives
// in the rotated value basis, is multiplied by R_V^T = P_br H U_V^T before it
// meets the BF16 partial.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) k_merge_plain(const float* __restrict__ partials, int hq_total, int nslots,
                                                     int nsplit, void* out, int out_dtype, float* lse) {
  const int hq = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
  const float* pb = partials + ((size_t)b * hq_total + hq) * nslots * kPartFloats;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, pb[s * kPartFloats]);
  float Ls = 0.f, A = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float m = pb[s * kPartFloats];
    if (m == -INFINITY) continue;
    const float w = exp2f(m - M);
    Ls = fmaf(pb[s * kPartFloats + 1], w, Ls);
    A = fmaf(pb[s * kPartFloats + 4 + c], w, A);
  }
  const float o = A / Ls;
  const size_t oi = ((size_t)b * hq_total + hq) * kD + c;
  if (out_dtype == OSCAR_OUT_FP32) static_cast<float*>(out)[oi] = o;
  else static_cast<__nv_bfloat16*>(out)[oi] = __float2bfloat16_rn(o);
  if (lse != nullptr && c == 0) lse[(size_t)b * hq_total + hq] = (M + log2f(Ls)) * 0.6931471805599453f;
}

// ---------------------------------------------------------------------------
// host launchers

int launch_decode_mma(const LayerView& lv, const DecodeWorkspace& ws, const DecodeArgs& a, float scale_log2,
                      cudaStream_t st);   // decode_mma.cu

template <int GQ>
static int launch_decode_gq(const LayerView& lv, const DecodeWorkspace& ws, const DecodeArgs& a, cudaStream_t st) {
  const float scale_log2 = a.sm_scale * kLog2e;
  if (!a.skip_qprep) {
    const int rc = launch_prologue(lv, ws, a.B, a.q, nullptr, nullptr, a.seq_lens, a.hist_pt, a.max_hist_pages,
                                   a.bf16_pt, a.sm_scale, st);
    if (rc != OSCAR_OK) return rc;
  }
  if (a.algo == OSCAR_DECODE_MMA || a.algo == OSCAR_DECODE_TC) {
    // the shared-prefix pages for all requests at once (if any), one fused launch for each request's
    // own history pages and the BF16 pages, then the merge kernel; the profiled span is the decode
    // launches (the events make them wait for the query prologue)
    if (a.ev0) cudaEventRecord(a.ev0, st);
    int rc = launch_decode_shared(lv, ws, a, st);
    if (rc == OSCAR_OK)
      rc = (a.algo == OSCAR_DECODE_TC && decode_tc_supported(lv)) ? launch_decode_tc(lv, ws, a, scale_log2, st)
                                                                   : launch_decode_mma(lv, ws, a, scale_log2, st);
    if (a.ev1) cudaEventRecord(a.ev1, st);
    if (rc != OSCAR_OK) return rc;
    return launch_merge(lv, ws, a.B, a.nsplit + a.nsplit_shared, a.nbf, a.out, a.out_dtype, a.lse, st);
  }
  if (a.ev0) cudaEventRecord(a.ev0, st);     // profiled span: the history kernel
  if (lv.meta_cb)
    k_int2_simt<GQ, true><<<dim3(a.nsplit, lv.hkv, a.B), 128, 0, st>>>(lv, ws, a.seq_lens, a.hist_pt, a.max_hist_pages,
                                                                       a.pages_per_split, scale_log2, a.len_add);
  else
    k_int2_simt<GQ, false><<<dim3(a.nsplit, lv.hkv, a.B), 128, 0, st>>>(lv, ws, a.seq_lens, a.hist_pt,
                                                                        a.max_hist_pages, a.pages_per_split,
                                                                        scale_log2, a.len_add);
  if (a.ev1) cudaEventRecord(a.ev1, st);
  k_bf16_seg<GQ><<<dim3(lv.hkv, a.B), 128, 0, st>>>(lv, ws, static_cast<const __nv_bfloat16*>(a.q), a.seq_lens,
                                                    a.bf16_pt, scale_log2, a.nsplit, a.len_add);
  if (cudaGetLastError() != cudaSuccess) return OSCAR_ERR_CUDA;
  return launch_merge(lv, ws, a.B, a.nsplit, 1, a.out, a.out_dtype, a.lse, st);
}

int launch_decode(const LayerView& lv, const DecodeWorkspace& ws, const DecodeArgs& a, cudaStream_t st) {
  if (a.B == 0) return OSCAR_OK;
  switch (lv.hq / lv.hkv) {
    case 1: return launch_decode_gq<1>(lv, ws, a, st);
    case 2: return launch_decode_gq<2>(lv, ws, a, st);
    case 4: return launch_decode_gq<4>(lv, ws, a, st);
    case 8: return launch_decode_gq<8>(lv, ws, a, st);
    default: return OSCAR_ERR_UNSUPPORTED;
  }
}

int launch_bf16_decode(int B, int hq, int hkv, const void* kv_pages, int num_pages, const void* q, const int* seq_lens,
                       const int* page_table, int max_pages, float sm_scale, void* out, int out_dtype, float* lse,
                       float* partials, int max_splits, int nsplit, int pps, int* status, cudaStream_t st) {
  if (B == 0) return OSCAR_OK;
  const int rc = launch_bf16_stream(B, hkv, hq, kv_pages, num_pages, q, seq_lens, page_table, max_pages, pps, nsplit,
                                    sm_scale * kLog2e, partials, max_splits, status, st);
  if (rc != OSCAR_OK) return rc;
  k_merge_plain<<<dim3(hq, B), 128, 0, st>>>(partials, hq, max_splits, nsplit, out, out_dtype, lse);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

int configure_mma_kernels();   // decode_mma.cu

int configure_decode_kernels() {
  if (configure_mma_kernels() != OSCAR_OK || configure_merge_kernel() != OSCAR_OK ||
      configure_tc_kernel() != OSCAR_OK || configure_bf16_stream() != OSCAR_OK)
    return OSCAR_ERR_CUDA;
  return configure_shared_kernel();
}

}  // namespace oscar
