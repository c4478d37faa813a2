// Shared device helpers for the MSA kernels (sm_103a): constants of the method, the device status
// word, asynchronous copies with L2 cache hints, and bf16 packing.  Every contraction of the
// library runs on the tcgen05 tensor cores (sm100.cuh); nothing here issues warp-level MMAs.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace msa {

constexpr int kBlock = 128;  // key block of the method
constexpr int kD = 128;      // head dim
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// device status word bits (first word of every workspace)
constexpr unsigned kStatusBadIndex = 1u;    // a block index out of range / not ascending
constexpr unsigned kStatusBadItems = 2u;    // work list larger than its reserved space
constexpr unsigned kStatusTimeout = 4u;     // a bounded device wait expired
constexpr unsigned kStatusInternal = 8u;    // a kernel's internal check failed (library bug)
// Words 8.. of the workspace's status area: work-item counters of the persistent kernels, each
// zeroed on the launch stream right before its kernel starts.
constexpr int kSchedAttnBwd = 8;
constexpr int kSchedProxyBwd = 9;
constexpr int kSchedAttnFwd = 10;
constexpr int kSchedProxyLse = 11;
constexpr int kSchedDenseFwd = 12;
// Word 16: the id of the first bounded wait that gave up, in kernels that record it (0: none).
constexpr int kStatusWhere = 16;

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; when !pred the destination is zero-filled and nothing
// is read (src must still be a valid pointer value).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred = true) {
  const uint32_t s = smem_u32(smem);
  const int sz = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(sz)
               : "memory");
}
// L2 eviction policies (createpolicy): data read many times (evict_last) or streamed once
// (evict_first), passed to the cache-hinted loads and stores below.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// cp_async16 with an L2 eviction policy.
__device__ __forceinline__ void cp_async16_hint(void* smem, const void* gmem, bool pred, uint64_t pol) {
  const uint32_t s = smem_u32(smem);
  const int sz = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n" ::"r"(s), "l"(gmem),
               "r"(sz), "l"(pol)
               : "memory");
}
// 16-byte global store / read-only load with an L2 eviction policy.
__device__ __forceinline__ void st_global_v4_hint(void* p, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;\n" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void st_global_f32_hint(float* p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;\n" ::"l"(p), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ uint4 ld_global_nc_v4_hint(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.b32 {%0, %1, %2, %3}, [%4], %5;\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
// Arrive on the mbarrier at `mbar` once every cp.async this thread issued so far has landed
// (counts as one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint64_t* mbar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(mbar))
               : "memory");
}
// 16-byte fp32 reduction predicated inside the instruction (no branch).
__device__ __forceinline__ void red_add_v4_if(bool pred, float* p, float4 v) {
  asm volatile(
      "{\n.reg .pred q;\nsetp.ne.b32 q, %5, 0;\n@q red.global.add.v4.f32 [%0], {%1, %2, %3, %4};\n}\n" ::"l"(p),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"((int)pred)
      : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Packed fp32 pairs (the sm_100 family's .f32x2 arithmetic): one instruction for two lanes, each
// lane rounded exactly like the scalar instruction (fma.rn / add.rn / mul.rn), so replacing a pair
// of scalar operations by one of these changes no result bit.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n.reg .b64 ra, rb, rc, rd;\nmov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %5};\n"
      "mov.b64 rc, {%6, %7};\nfma.rn.f32x2 rd, ra, rb, rc;\nmov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 r;
  asm("{\n.reg .b64 ra, rb, rd;\nmov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %5};\n"
      "add.rn.f32x2 rd, ra, rb;\nmov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 r;
  asm("{\n.reg .b64 ra, rb, rd;\nmov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %5};\n"
      "mul.rn.f32x2 rd, ra, rb;\nmov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
// Three-input maximum (sm_100 family); the maximum does not depend on the order of its inputs.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

}  // namespace msa
