// np_common.cuh -- device helpers shared by the kernels of libnp_paged.so:
// mbarrier and bulk-copy (TMA) inline PTX, bounded waits, storage-type
// widening, error flags.  sm_103a only.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the library never links libcuda)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "np_paged.h"

namespace npk {

// ---------------------------------------------------------------- errors --
__device__ __forceinline__ void set_flag(int32_t* err, int32_t bit) {
  if (err != nullptr) atomicOr(err, bit);
}

// ----------------------------------------------------------------- time ---
// A pipeline wait gives up after this many SM clock cycles (about 1 s at the
// GB300's 2.07 GHz maximum clock; nothing legitimate takes more than
// microseconds).  clock64 is the SM's own counter: cheap to read, unlike the
// global timer.
constexpr long long kWaitLimitCycles = 2000000000ll;

// ------------------------------------------------------------- mbarrier ---
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits until the phase with the given parity has completed.  Bounded: gives
// up (returns false) when *abort becomes non-zero or after `limit` cycles
// (kWaitLimitCycles unless a self-test asks for less), in which case it sets
// *abort itself so every other waiter in the block stops.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (clock64() - t0 > limit) {
        *abort = 1;
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag (used to drain copies in flight).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity) && clock64() - t0 < kWaitLimitCycles) {
  }
}

// ----------------------------------------------------- bulk copy (TMA) ----
// L2 policy for streamed K/V: read once, evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes`
// transactions on `bar`.  src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                        uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Tiled 3-D TMA load: the box at coordinates (c0, c1, c2) of `map` into this
// CTA's shared memory, completing its bytes on `bar`.  c0 * element size must
// be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t c0,
                                           int32_t c1, int32_t c2, uint32_t bar,
                                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
      : "memory");
}

// 4-D tiled copy (coordinates innermost first) into this CTA's shared memory.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int32_t c0,
                                           int32_t c1, int32_t c2, int32_t c3, uint32_t bar,
                                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
      "l"(policy)
      : "memory");
}

// ------------------------------------------------------ row stores --------
// Plain stores of result rows (shared or global memory).
struct PlainStore {
  __device__ __forceinline__ void operator()(float* p, float v) const { *p = v; }
  __device__ __forceinline__ void v4(float* p, const float* v) const {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};

// Global stores of rows that a later kernel of the same step reads back
// (the balanced read's cut-row partials and merge descriptors), with an L2
// evict-last hint: the read streams GBs through L2 (evict-first) after
// writing them, and without the hint the merge finds them in DRAM.
struct L2KeepStore {
  uint64_t pol;
  __device__ __forceinline__ static L2KeepStore make() {
    L2KeepStore s;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(s.pol));
    return s;
  }
  __device__ __forceinline__ void operator()(float* p, float v) const {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol)
                 : "memory");
  }
  __device__ __forceinline__ void v4(float* p, const float* v) const {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p),
                 "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "l"(pol)
                 : "memory");
  }
  __device__ __forceinline__ void i4(int4* p, int4 v) const {
    asm volatile("st.global.L2::cache_hint.v4.s32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
  }
};

// ----------------------------------------------------------- arithmetic ---
// 2^x (PTX ex2.approx, flush-to-zero); ex2(-inf) = +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------- storage types ----
// Widening of 16-byte / 8-byte vectors of the storage type to fp32.
// bf16 is the top half of an fp32, so widening is a shift or a mask.
template <typename T>
struct Storage;

template <>
struct Storage<float> {
  static constexpr int kBytes = 4;
  static constexpr np_dtype kDtype = NP_F32;
  // n elements (8, 4 or 2) from a 16- or 8-byte aligned address
  template <int N>
  __device__ __forceinline__ static void load(const float* p, float* x) {
    if constexpr (N == 8) {
      load<4>(p, x);
      load<4>(p + 4, x + 4);
    } else if constexpr (N == 4) {
      float4 v = *reinterpret_cast<const float4*>(p);
      x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else if constexpr (N == 2) {
      float2 v = *reinterpret_cast<const float2*>(p);
      x[0] = v.x; x[1] = v.y;
    } else {
      static_assert(N == 1, "vector width");
      x[0] = *p;
    }
  }
  template <int N>
  __device__ __forceinline__ static void store(float* p, const float* x) {
    if constexpr (N == 8) {
      store<4>(p, x);
      store<4>(p + 4, x + 4);
    } else if constexpr (N == 4) {
      *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    } else if constexpr (N == 2) {
      *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
    } else {
      static_assert(N == 1, "vector width");
      *p = x[0];
    }
  }
};

__device__ __forceinline__ void widen_bf16x2(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

template <>
struct Storage<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  static constexpr np_dtype kDtype = NP_BF16;
  template <int N>
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* x) {
    if constexpr (N == 8) {
      uint4 v = *reinterpret_cast<const uint4*>(p);
      widen_bf16x2(v.x, x[0], x[1]);
      widen_bf16x2(v.y, x[2], x[3]);
      widen_bf16x2(v.z, x[4], x[5]);
      widen_bf16x2(v.w, x[6], x[7]);
    } else if constexpr (N == 4) {
      uint2 v = *reinterpret_cast<const uint2*>(p);
      widen_bf16x2(v.x, x[0], x[1]);
      widen_bf16x2(v.y, x[2], x[3]);
    } else if constexpr (N == 2) {
      uint32_t v = *reinterpret_cast<const uint32_t*>(p);
      widen_bf16x2(v, x[0], x[1]);
    } else {
      static_assert(N == 1, "vector width");
      x[0] = __bfloat162float(*p);
    }
  }
  // fp32 -> bf16 round-to-nearest-even
  template <int N>
  __device__ __forceinline__ static void store(__nv_bfloat16* p, const float* x) {
    if constexpr (N >= 2) {
      static_assert(N % 2 == 0 && N <= 8, "vector width");
      uint32_t w[N / 2];
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&h);
      }
      if constexpr (N == 8) {
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
      } else if constexpr (N == 4) {
        *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
      } else {
        *reinterpret_cast<uint32_t*>(p) = w[0];
      }
    } else {
      *p = __float2bfloat16_rn(x[0]);
    }
  }
};

}  // namespace npk
