// Optional kernel timeline (oscar_trace_timeline): thread 0 of every CTA of a
// traced kernel claims one record and stamps it with %globaltimer on entry and
// when it leaves the kernel body. Costs one predicated branch when off.
#pragma once

#include "common.cuh"
#include "tma.cuh"

namespace oscar {

enum TimelineKind : int {
  kTlAppend = 1, kTlQprep = 2, kTlDecodeMma = 3, kTlMerge = 4, kTlInt2Simt = 5, kTlBf16Seg = 6, kTlPrefill = 7,
  kTlDecodeShared = 8
};

// record i lives at timeline[4 + 4 i]: {kind | layer << 8 | sm << 24 | linear CTA << 32, start, end, mark};
// timeline[0] counts the records claimed. The record address is kept in
// shared memory (thread 0 reads it back), not in a register for the kernel's
// whole life.
__device__ __forceinline__ unsigned long long* volatile& timeline_slot() {
  __shared__ unsigned long long* volatile slot;
  return slot;
}

struct TimelineSpan {
  __device__ __forceinline__ TimelineSpan(const LayerView& lv, int kind) {
    if (threadIdx.x != 0) return;
    unsigned long long* rec = nullptr;
    if (lv.timeline != nullptr) {
      const unsigned long long i = atomicAdd(lv.timeline, 1ull);
      if (i < (unsigned long long)lv.timeline_cap) {
        const unsigned long long cta = blockIdx.x + gridDim.x * (blockIdx.y + (unsigned long long)gridDim.y * blockIdx.z);
        rec = lv.timeline + 4 + 4 * i;
        rec[0] = (unsigned long long)kind | ((unsigned long long)(lv.layer & 0xffff) << 8) |
                 ((unsigned long long)(sm_id() & 0xff) << 24) | (cta << 32);
        rec[1] = global_ns();
        rec[3] = 0;
      }
    }
    timeline_slot() = rec;
  }
  // an intermediate time of the kernel's choosing (the programmatic wait returning); thread 0 only
  __device__ __forceinline__ void mark() {
    if (threadIdx.x != 0) return;
    unsigned long long* rec = timeline_slot();
    if (rec != nullptr) rec[3] = global_ns();
  }
  __device__ __forceinline__ ~TimelineSpan() {
    if (threadIdx.x != 0) return;
    unsigned long long* rec = timeline_slot();
    if (rec != nullptr) rec[2] = global_ns();
  }
};

}  // namespace oscar
