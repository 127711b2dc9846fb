// Device helpers shared by the kernels of libpagedkv: the device error record,
// inline-PTX wrappers for mbarrier and the bulk (TMA) global->shared copy, and
// 16-byte half/bfloat16 <-> fp32 conversions.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include <cstdint>

#include "pagedkv.h"

namespace pagedkv {

constexpr uint32_t kFullMask = 0xffffffffu;
// Upper bound on any spin wait inside a kernel.  A legitimate wait here is a few
// microseconds (one bulk copy, or one consumer step); one second means the
// machine is wedged, so the kernel records PA_ERR_TIMEOUT and returns.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// ---------------------------------------------------------------- error record
__device__ __forceinline__ void report_error(int32_t* rec, int code, long long index,
                                             long long value) {
  if (rec == nullptr) return;
  if (atomicCAS(reinterpret_cast<int*>(rec), 0, code) == 0) {
    rec[2] = static_cast<int32_t>(index);
    rec[3] = static_cast<int32_t>(value);
  }
  atomicAdd(reinterpret_cast<int*>(rec) + 1, 1);
}

// ------------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make mbarrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// True once the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for a phase, giving up after `limit_ns` of wall time.  Returns false on
// timeout.  The timer is only read every 16 failed polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// ------------------------------------------------------- bulk (TMA) 1-D copy
// L2 policy for data read exactly once (K/V rows): evict first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Global -> shared bulk copy that signals `bar` with complete_tx.  Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// ------------------------------------------------------------ conversions
struct F16 {
  using T = __half;
};
struct BF16 {
  using T = __nv_bfloat16;
};

// Eight packed 16-bit values -> eight floats (exact).
__device__ __forceinline__ void to_float8(const uint4& u, float (&f)[8], BF16) {
  // A bfloat16 is the upper half of a binary32: shift it into place.
  f[0] = __uint_as_float(u.x << 16);
  f[1] = __uint_as_float(u.x & 0xffff0000u);
  f[2] = __uint_as_float(u.y << 16);
  f[3] = __uint_as_float(u.y & 0xffff0000u);
  f[4] = __uint_as_float(u.z << 16);
  f[5] = __uint_as_float(u.z & 0xffff0000u);
  f[6] = __uint_as_float(u.w << 16);
  f[7] = __uint_as_float(u.w & 0xffff0000u);
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t bits) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = bits;
  return __half22float2(h);
}

__device__ __forceinline__ void to_float8(const uint4& u, float (&f)[8], F16) {
  float2 a = half2_bits_to_float2(u.x), b = half2_bits_to_float2(u.y);
  float2 c = half2_bits_to_float2(u.z), d = half2_bits_to_float2(u.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, int dtype) {
  if (dtype == PA_BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Store n (2, 4 or 8) consecutive fp32 values as `dtype` at element offset
// `elem` of `out`.  The address is a multiple of n elements.
template <int N>
__device__ __forceinline__ void store_out(void* out, size_t elem, const float* v, int dtype) {
  if (dtype == PA_F32) {
    float* o = static_cast<float*>(out) + elem;
    if constexpr (N % 4 == 0) {
#pragma unroll
      for (int j = 0; j < N; j += 4)
        *reinterpret_cast<float4*>(o + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < N; j += 2) *reinterpret_cast<float2*>(o + j) = make_float2(v[j], v[j + 1]);
    }
  } else {
    uint16_t* o = static_cast<uint16_t*>(out) + elem;
    if constexpr (N == 8) {
      *reinterpret_cast<uint4*>(o) = make_uint4(pack2(v[0], v[1], dtype), pack2(v[2], v[3], dtype),
                                                pack2(v[4], v[5], dtype), pack2(v[6], v[7], dtype));
    } else if constexpr (N == 4) {
      *reinterpret_cast<uint2*>(o) = make_uint2(pack2(v[0], v[1], dtype), pack2(v[2], v[3], dtype));
    } else {
      *reinterpret_cast<uint32_t*>(o) = pack2(v[0], v[1], dtype);
    }
  }
}

// Host-side helpers -------------------------------------------------------
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Named NVTX range over a C-ABI call, so the library's calls show up in
// Nsight timelines; a push/pop costs a few ns when no tool is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace pagedkv
