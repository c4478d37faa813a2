// Blackwell (sm_100 family, here sm_103a) tensor-core building blocks in inline PTX:
// tensor memory (TMEM) allocation and loads, tcgen05.mma issue/commit, mbarriers with bounded
// waits, and shared-memory matrix descriptors for the 128-byte-swizzled canonical layout.
//
// Shared-memory operand layout ("SW128"): a tile of R rows x 64 bf16 (128 bytes per row) stored
// row after row, 8-row atoms of 1024 bytes, 16-byte chunk c of row r placed at chunk
// (c XOR (r mod 8)).  A 128-wide tile is two such 64-wide column panels, one after the other.
// The same bytes serve as
//   * a K-major operand when rows index M (or N) and the 64 columns index K, and
//   * an MN-major operand when rows index K and the 64 columns index M (or N);
// only the descriptor differs (see desc_kmajor / desc_mnmajor).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace msa {
namespace sm100 {

// ------------------------------------------------------------------ SW128 layout helpers
// Byte offset of element (row, col) inside one 64-column panel of the SW128 layout.
__device__ __forceinline__ uint32_t sw128_offset(int row, int col) {
  const int chunk = (col >> 3) ^ (row & 7);
  return (uint32_t)(row * 128 + (chunk << 4) + ((col & 7) << 1));
}
// Byte offset of the 16-byte chunk `c16` (0..7) of `row` inside a panel.
__device__ __forceinline__ uint32_t sw128_chunk(int row, int c16) {
  return (uint32_t)(row * 128 + (((c16 ^ (row & 7)) & 7) << 4));
}

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor: start address, leading / stride byte offsets (>> 4), the
// fixed version field (1) of this architecture, and the 128-byte swizzle mode (2).
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // version
  d |= (uint64_t)2 << 61;  // SWIZZLE_128B
  return d;
}
// K-major operand, K step `ks` (16 elements) of a tile whose panels hold `rows` rows each.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile_saddr, int rows, int ks) {
  const uint32_t a = tile_saddr + (uint32_t)((ks >> 2) * rows * 128 + (ks & 3) * 32);
  return make_desc(a, 16, 1024);
}
// MN-major operand, K step `ks` (16 rows) of a tile with `rows` (= K extent) rows per panel;
// consecutive 64-wide MN panels are rows*128 bytes apart.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile_saddr, int rows, int ks) {
  const uint32_t a = tile_saddr + (uint32_t)(ks * 16 * 128);
  return make_desc(a, (uint32_t)(rows * 128), 1024);
}

// Instruction descriptor for kind::f16 with bf16 A/B, fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                                   // D format: f32
         | (1u << 7)                                 // A format: bf16
         | (1u << 10)                                // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15)            // A major
         | ((b_mn_major ? 1u : 0u) << 16)            // B major
         | ((uint32_t)(N >> 3) << 17)                // N / 8
         | ((uint32_t)(M >> 4) << 24);               // M / 16
}

// ------------------------------------------------------------------ TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Named barrier `id` (1..15) over `nthreads` threads of whole, converged warps.  Callers keep
// every participating warp on the same sequence of these barriers (no early exits between them).
__device__ __forceinline__ void bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// Make generic-proxy shared-memory writes (st.shared, cp.async) visible to the tensor core.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// 32 lanes x 32 columns of 32-bit: thread i of the warp gets lane (base lane + i), 32 columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// 32 lanes x 32 columns of 32-bit stores (thread i writes lane base + i).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
               "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// ------------------------------------------------------------------ MMA
// D[tmem] (+)= A[smem] * B[smem]; issued by one thread.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                      uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]: A is M x K bf16 in tensor memory, lane = row, two K elements
// per 32-bit column (K step ks starts at column 8 * ks).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                      uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}
// Arrive on an mbarrier once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          static_cast<uint32_t>(__cvta_generic_to_shared(mbar)))
      : "memory");
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(mbar))),
               "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* mbar) {
  asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(mbar)))
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* mbar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(mbar))), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: spins on try_wait (which itself suspends the thread until the phase completes or
// a short hardware time limit passes) and gives up after `limit_ns` of wall time (legitimate
// waits here last microseconds), setting the timeout bit (4) of the device status word.
// Every wait in this library is bounded and callers leave their loops on a timeout, so a logic
// error can never hang the GPU.
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t parity, unsigned* err,
                                          uint64_t limit_ns = 200000000ull) {
  if (mbar_try_wait(mbar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(mbar, parity)) return true;
    if ((i & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) break;
  }
  if (err) atomicOr(err, 4u);
  return false;
}

// Warp-collective form of mbar_wait for roles in which every lane waits: the result is the AND
// over the warp, so the lanes leave (or continue) together.  Warp-collective instructions that
// follow (tcgen05.ld / st, __syncwarp) must never run with part of a warp.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* mbar, uint32_t parity, unsigned* err) {
  const bool ok = mbar_wait(mbar, parity, err);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------ TMA (bulk tensor copies)
__device__ __forceinline__ void mbar_expect_tx(uint64_t* mbar, uint32_t bytes) {
  asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(mbar))),
               "r"(bytes)
               : "memory");
}
// Tiled 2D / 3D loads global -> shared (SW128 layout set by the tensor map); completion is
// reported to `mbar` as transaction bytes.  The innermost coordinate must be a multiple of 8
// elements (16 bytes) -- every call here passes 0 or 64.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int c0, int c1,
                                            uint64_t* mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];\n" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
      "l"(tmap), "r"(c0), "r"(c1), "r"(static_cast<uint32_t>(__cvta_generic_to_shared(mbar)))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int c0, int c1, int c2,
                                            uint64_t* mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4}], [%5];\n" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2),
      "r"(static_cast<uint32_t>(__cvta_generic_to_shared(mbar)))
      : "memory");
}
// Row gather: four rows r0..r3 (any order, any distance) of a 2D tensor whose map has a box
// of 64 columns x 1 row; the rows land one after the other at dst (4 x 128 bytes, swizzled like
// rows of a tile at that shared-memory address).  c0 is the column (0 or 64).
__device__ __forceinline__ void tma_gather4(void* dst, const void* tmap, int c0, int r0, int r1,
                                            int r2, int r3, uint64_t* mbar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;\n" ::"r"(
          static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
      "l"(tmap), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
      "r"(static_cast<uint32_t>(__cvta_generic_to_shared(mbar))), "l"(policy)
      : "memory");
}
// Plain (untiled) bulk copy global -> shared of `bytes` bytes (both addresses 16-byte aligned,
// size a multiple of 16), completion reported to `mbar` as transaction bytes.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
      "l"(src), "r"(bytes), "r"(static_cast<uint32_t>(__cvta_generic_to_shared(mbar)))
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(tmap) : "memory");
}

// Round a dynamic shared-memory pointer up to the 1024-byte alignment the SW128 atoms need.
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  return p + (((a + 1023u) & ~1023u) - a);
}

}  // namespace sm100
}  // namespace msa
