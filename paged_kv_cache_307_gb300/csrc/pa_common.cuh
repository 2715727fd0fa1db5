// pa_common.cuh — shared device helpers for libpa (sm_103a).
//
// Inline PTX for the Blackwell async-copy path: mbarrier init/arrive/wait,
// TMA tensor loads (cp.async.bulk.tensor) completing on an mbarrier, and a
// bounded wait that gives up after a wall-clock limit instead of spinning
// forever.  Every translation unit keeps its own sticky status word and
// exposes a host function that fetches and clears it.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// A wait that has not completed after this long is treated as a pipeline
// failure: the kernel records PA_DEV_TIMEOUT and winds down.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Returns
// false if it has not completed within limit_ns.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}
// The library's pipeline wait: kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, kWaitLimitNs);
}

// 4-D TMA tile load global -> shared, completion signalled on `bar` as
// transaction bytes.  Coordinates are innermost first.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Untiled bulk copy global -> shared completing on an mbarrier; both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tensor core) before the memory is handed back to it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `nthreads` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 16-byte global loads that bypass L1 allocation (streamed once).
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// bf16 pair (packed in a 32-bit word, low half first) -> two floats.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kBytes = 4;
  static constexpr int kPerChunk = 4;   // elements in 16 bytes
  __device__ __forceinline__ static void unpack(const uint4& c, float* f) {
    f[0] = __uint_as_float(c.x); f[1] = __uint_as_float(c.y);
    f[2] = __uint_as_float(c.z); f[3] = __uint_as_float(c.w);
  }
  __device__ __forceinline__ static float load1(const float* p) { return *p; }
  __device__ __forceinline__ static void store1(float* p, float v) { *p = v; }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  static constexpr int kPerChunk = 8;
  __device__ __forceinline__ static void unpack(const uint4& c, float* f) {
    f[0] = bf16lo(c.x); f[1] = bf16hi(c.x); f[2] = bf16lo(c.y); f[3] = bf16hi(c.y);
    f[4] = bf16lo(c.z); f[5] = bf16hi(c.z); f[6] = bf16lo(c.w); f[7] = bf16hi(c.w);
  }
  __device__ __forceinline__ static float load1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  __device__ __forceinline__ static void store1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

// Packed fp32 pairs: one 64-bit register, the f32x2 instructions (two lanes
// of fma, add or mul per instruction, each lane rounded as the scalar
// instruction would round it).
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Tag type for e4m3 codes in a K/V pool (one byte per element).
struct fp8e4m3 {
  uint8_t bits;
};
// Four e4m3 codes (byte i = element i) to two f16x2 values (elements 0,1
// and 2,3), exactly: every e4m3 value is an f16 value.  The 32-bit word is
// split into its 16-bit halves and each is converted by one instruction.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}
// An f16x2 value to two floats, exactly.
__device__ __forceinline__ void f16x2_to_float2(uint32_t h, float& lo, float& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h));
}
template <> struct Elem<fp8e4m3> {
  static constexpr int kBytes = 1;
  static constexpr int kPerChunk = 16;
  __device__ __forceinline__ static void unpack(const uint4& c, float* f) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t h01, h23;
      e4m3x4_to_f16x2x2(w[i], h01, h23);
      f16x2_to_float2(h01, f[4 * i], f[4 * i + 1]);
      f16x2_to_float2(h23, f[4 * i + 2], f[4 * i + 3]);
    }
  }
};

inline int elem_bytes(pa_dtype dt) { return dt == PA_F32 ? 4 : dt == PA_FP8_E4M3 ? 1 : 2; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool supported_head_dim(int d) { return d == 32 || d == 64 || d == 128; }
inline bool supported_block_size(int bs) { return bs == 4 || bs == 8 || bs == 16 || bs == 32; }

// Host: number of SMs on the current device (cached per device).
int device_sm_count();


// Host: encode a tiled tensor map of rank <= 5 (dims/box innermost first,
// strides in bytes for dims 1..rank-1), bf16 or fp32, optionally with the
// 128-byte shared-memory swizzle.  Returns false on failure.
bool encode_map(CUtensorMap* map, const void* base, pa_dtype dt, int rank, const uint64_t* dims,
                const uint64_t* strides, const uint32_t* box, bool swizzle128);

// Host: record the text of the last host-side failure (per thread); read
// back through pa_last_host_error().
void note_host_error(const char* what);
// Host: true if `e` is cudaSuccess, otherwise records "<what>: <error>".
bool ck(cudaError_t e, const char* what);
// Host: raise `kernel`'s dynamic shared-memory limit to the device opt-in
// maximum (once per kernel and device).
bool raise_smem_limit(const void* kernel, int dev);

// Launch `kernel` on `stream` as a programmatic dependent of the kernel before
// it (it may be scheduled once that grid has started; it must wait with
// griddepcontrol.wait before reading that grid's results), unless the stream
// is being captured, where a plain launch is kept (graph replay measured
// slower with the programmatic edge).  Falls back to a plain launch when the
// runtime does not accept the attribute.
cudaError_t launch_after(const void* kernel, dim3 grid, dim3 block, void** args, cudaStream_t stream);

// Per-translation-unit status fetch (returns the sticky word and clears it).
unsigned fetch_status_cache_ops();
unsigned fetch_status_decode();
unsigned fetch_status_decode_fp8();
unsigned fetch_status_shared();
unsigned fetch_status_prefill();
unsigned fetch_status_selftest();

}  // namespace pa
