// Device helpers shared by the two tcgen05 decode kernels: the walk over a worker's pages, 32-byte
// non-coherent loads, shared-memory stores, and bounded waits that report a timeout in the plan's
// status word instead of hanging.
#pragma once

#include <cstdint>

#include "qkvp_internal.h"
#include "tc_ptx.cuh"

namespace qkvp {
namespace kern {

// Walks a worker's (segment, page) sequence.
struct Cursor {
  int si, se, j;
  Segment seg;
  __device__ void begin(const DecodeArgs& a, int s0, int s1) {
    si = s0; se = s1; j = 0;
    if (si < se) seg = a.segs[si];
  }
  __device__ bool done() const { return si >= se; }
  __device__ void next(const DecodeArgs& a) {
    if (++j >= seg.num_pages) { j = 0; if (++si < se) seg = a.segs[si]; }
  }
  __device__ int valid() const { return min(kPage, seg.num_tokens - j * kPage); }
  __device__ int64_t page(const DecodeArgs& a) const { return a.kv_indices[seg.page_begin + j]; }
};

// A page index outside the pool reads as an empty page.
__device__ __forceinline__ bool page_ok(const DecodeArgs& a, int64_t page) { return page >= 0 && page < a.num_pages; }

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// 32 bytes from global memory through the non-coherent path (the address must be 32-byte aligned).
__device__ __forceinline__ void ldg_nc32(const void* p, uint32_t (&v)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "l"(p));
}

// The same store without a compiler memory barrier: later global loads may be issued before it. Only
// for shared memory that no ordinary load reads (operands the tensor cores read after a proxy fence).
__device__ __forceinline__ void sts128_relaxed(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// The CTA's mbarriers (8 bytes each from `bars`), its abort flag and the plan's status word.
struct Sync {
  uint32_t bars;
  volatile int* abort;
  int* status;
  __device__ uint32_t bar(uint32_t i) const { return bars + 8 * i; }
  // Bounded wait for the phase of `parity` of barrier i (acquire at cluster scope if `cluster`). After
  // ~2^31 cycles it sets `code` in the status word and the abort flag, which ends every other wait of
  // the CTA early; false then.
  __device__ bool wait(uint32_t i, uint32_t parity, bool cluster = false, int code = 1) const {
    const uint32_t b = bar(i);
    if (cluster ? tc::mbar_try_wait_cluster(b, parity) : tc::mbar_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    for (int n = 0;; ++n) {
      if (cluster ? tc::mbar_try_wait_cluster(b, parity) : tc::mbar_try_wait(b, parity)) return true;
      if ((n & 255) == 0) {
        if (*abort) return false;
        if (clock64() - t0 > (1ll << 31)) {
          *abort = 1;
          atomicOr(status, code);
          return false;
        }
      }
    }
  }
};

// Bounded wait until the counter at `addr` reaches `target` (acquire: what was written before the
// counter was raised is visible afterwards); a timeout sets `code` like Sync::wait.
__device__ __forceinline__ bool wait_counter(const Sync& sy, uint32_t addr, uint32_t target, int code) {
  if (tc::ld_acquire_u32(addr) >= target) return true;
  const long long t0 = clock64();
  for (int n = 0;; ++n) {
    if (tc::ld_acquire_u32(addr) >= target) return true;
    if ((n & 255) == 0) {
      if (*sy.abort) return false;
      if (clock64() - t0 > (1ll << 31)) {
        *sy.abort = 1;
        atomicOr(sy.status, code);
        return false;
      }
    }
  }
}

}  // namespace kern
}  // namespace qkvp
