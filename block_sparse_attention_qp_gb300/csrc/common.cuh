// Shared device helpers for the MSA kernels (sm_103a).
//
// Tile conventions used by every attention-shaped kernel here:
//   * head dim D = 128 and key block = 128 tokens (the method's only supported shapes);
//   * bf16 tiles in shared memory are row-major with a padded row of kLd elements (272 bytes),
//     which keeps 8-row ldmatrix accesses free of bank conflicts;
//   * warp-level products use the m16n8k16 bf16 tensor-core instruction with fp32 accumulate;
//     an accumulator "acc[N/8][4]" holds a 16 x N fp32 tile in the instruction's C layout:
//     acc[j][0..1] -> row lane/4,     columns 8j + 2(lane%4) + {0,1}
//     acc[j][2..3] -> row lane/4 + 8, same columns.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace msa {

constexpr int kBlock = 128;  // key block of the method
constexpr int kD = 128;      // head dim
constexpr int kLd = kD + 8;  // padded bf16 row in shared memory
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// device status word bits (first word of every workspace)
constexpr unsigned kStatusBadIndex = 1u;    // a block index out of range / not ascending
constexpr unsigned kStatusBadItems = 2u;    // work list larger than its reserved space
constexpr unsigned kStatusTimeout = 4u;     // a bounded device wait expired
// Words 8.. of the workspace's status area: work-item counters of the persistent kernels, each
// zeroed on the launch stream right before its kernel starts.
constexpr int kSchedAttnBwd = 8;
constexpr int kSchedProxyBwd = 9;
constexpr int kSchedAttnFwd = 10;

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

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int NT>
__device__ __forceinline__ void zero_acc(float (&acc)[NT][4]) {
#pragma unroll
  for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
}

// acc (16 x N) += A (16 x K, smem row-major, lda) * Bt^T, Bt is [N][K] row-major (ldb).
template <int N, int K>
__device__ __forceinline__ void warp_gemm_abt(float (&acc)[N / 8][4], const bf16* a, int lda,
                                              const bf16* bt, int ldb, int lane) {
#pragma unroll
  for (int kk = 0; kk < K; kk += 16) {
    uint32_t af[4];
    ldsm_x4(af, a + (lane % 16) * lda + kk + (lane / 16) * 8);
#pragma unroll
    for (int nn = 0; nn < N; nn += 16) {
      uint32_t bfr[4];
      ldsm_x4(bfr, bt + (nn + (lane % 8) + (lane / 16) * 8) * ldb + kk + ((lane / 8) % 2) * 8);
      mma16816(acc[nn / 8], af, bfr[0], bfr[1]);
      mma16816(acc[nn / 8 + 1], af, bfr[2], bfr[3]);
    }
  }
}

// acc (16 x N) += A (16 x K, smem row-major, lda) * B, B is [K][N] row-major (ldb).
template <int N, int K>
__device__ __forceinline__ void warp_gemm_ab(float (&acc)[N / 8][4], const bf16* a, int lda,
                                             const bf16* b, int ldb, int lane) {
#pragma unroll
  for (int kk = 0; kk < K; kk += 16) {
    uint32_t af[4];
    ldsm_x4(af, a + (lane % 16) * lda + kk + (lane / 16) * 8);
#pragma unroll
    for (int nn = 0; nn < N; nn += 16) {
      uint32_t bfr[4];
      ldsm_x4_t(bfr, b + (kk + (lane % 8) + ((lane / 8) % 2) * 8) * ldb + nn + (lane / 16) * 8);
      mma16816(acc[nn / 8], af, bfr[0], bfr[1]);
      mma16816(acc[nn / 8 + 1], af, bfr[2], bfr[3]);
    }
  }
}

// acc (16 x N) += A * B with A given as register fragments af[K/16][4] (from a C-layout tile),
// B is [K][N] row-major in smem (ldb).
template <int N, int K>
__device__ __forceinline__ void warp_gemm_rb(float (&acc)[N / 8][4], const uint32_t (&af)[K / 16][4],
                                             const bf16* b, int ldb, int lane) {
#pragma unroll
  for (int kk = 0; kk < K; kk += 16) {
#pragma unroll
    for (int nn = 0; nn < N; nn += 16) {
      uint32_t bfr[4];
      ldsm_x4_t(bfr, b + (kk + (lane % 8) + ((lane / 8) % 2) * 8) * ldb + nn + (lane / 16) * 8);
      mma16816(acc[nn / 8], af[kk / 16], bfr[0], bfr[1]);
      mma16816(acc[nn / 8 + 1], af[kk / 16], bfr[2], bfr[3]);
    }
  }
}

// acc (16 x N) += X^T (rows m0..m0+15 of X^T) * B, X is [K][M] row-major (ldx), B is [K][N]
// row-major (ldb).  Used for dV = P^T dO, dK = dS^T Q, dKp = dz^T Qp.
template <int N, int K>
__device__ __forceinline__ void warp_gemm_atb(float (&acc)[N / 8][4], const bf16* x, int ldx,
                                              int m0, const bf16* b, int ldb, int lane) {
#pragma unroll
  for (int kk = 0; kk < K; kk += 16) {
    uint32_t af[4];
    ldsm_x4_t(af, x + (kk + (lane % 8) + (lane / 16) * 8) * ldx + m0 + ((lane / 8) % 2) * 8);
#pragma unroll
    for (int nn = 0; nn < N; nn += 16) {
      uint32_t bfr[4];
      ldsm_x4_t(bfr, b + (kk + (lane % 8) + ((lane / 8) % 2) * 8) * ldb + nn + (lane / 16) * 8);
      mma16816(acc[nn / 8], af, bfr[0], bfr[1]);
      mma16816(acc[nn / 8 + 1], af, bfr[2], bfr[3]);
    }
  }
}

// Convert a 16 x K fp32 C-layout tile into A-operand fragments (bf16) for a following product.
template <int K>
__device__ __forceinline__ void c_to_a(uint32_t (&af)[K / 16][4], const float (&c)[K / 8][4]) {
#pragma unroll
  for (int j = 0; j < K / 16; ++j) {
    af[j][0] = pack_bf16(c[2 * j][0], c[2 * j][1]);
    af[j][1] = pack_bf16(c[2 * j][2], c[2 * j][3]);
    af[j][2] = pack_bf16(c[2 * j + 1][0], c[2 * j + 1][1]);
    af[j][3] = pack_bf16(c[2 * j + 1][2], c[2 * j + 1][3]);
  }
}

// Load `rows` rows of 128 bf16 from global rows given by a per-row pointer function into a
// padded smem tile; rows with a null pointer are zero-filled.
template <typename RowPtr>
__device__ __forceinline__ void load_rows_async(bf16* s, int rows, RowPtr rowptr, int tid,
                                                int nthreads, const void* any_valid) {
  for (int c = tid; c < rows * 16; c += nthreads) {
    const int r = c >> 4, ch = c & 15;
    const bf16* g = rowptr(r);
    cp_async16(s + r * kLd + ch * 8, g ? (const void*)(g + ch * 8) : any_valid, g != nullptr);
  }
}

}  // namespace msa
