// Backward on the tcgen05 tensor cores (blog, "Backward" and "KL Divergence Loss"):
//   rowdot_kernel     row data {LSE log2 e, D = rowsum(dO * O)} of every query row
//   attn_bwd_kernel   main-attention gradients dQ, dK, dV and the teacher pbar
//   proxy_bwd_kernel  proxy gradients dQp, dKp of the KL term, from pbar
//
// Work items (shared by both kernels): one 128-key block n of group g and up to 512 tokens that
// use it (from the inverted block map; in warmup mode every token t >= 128 n), all from one
// sequence chunk.  Lists run chunk-major and blocks take items in list order from a shared
// counter, so the dQ / dQp rows that concurrent items update belong to one chunk of the sequence.
//
// attn_bwd_kernel keeps the block's K and V in shared memory and its dK, dV accumulators in tensor
// memory while it streams tiles of 64/G tokens x G query heads (64 rows) through three Q / dO
// slots (S^T and dP^T double buffered in tensor memory):
//   phase 1 (tensor core)  S^T = K Q^T,  dP^T = V dO^T                       (keys x rows, fp32)
//   softmax (4 warps, thread = key)
//                          P^T  = exp(scale S^T - LSE_row)       -> tensor memory (bf16)
//                          dS^T = P^T (dP^T - D_row)             -> shared memory (bf16)
//                          teacher pbar = mean over the token's G heads of P -> global (fp16)
//   phase 2 (tensor core)  dV += P^T dO,  dK += dS^T Q,  dQ^T = K^T dS^T
//   epilogue               dQ^T -> fp32 rows staged in the tile's own slot; a reducer thread adds
//                          each token's G rows into dQ with one bulk TMA reduction
//   item end               dK (x scale), dV -> fp32 atomics
// proxy_bwd_kernel streams the same items in groups of 64 tokens:
//   z^T = Kp Qp^T;  dz = kl_grad/(B S Hp) (exp(scale z - LSE_px) - pbar)   (the blog's closed
//   form; the teacher is a constant, so no KL term reaches dQ, dK, dV)
//   dKp += dz^T Qp (tensor memory, per item),  dQp^T = Kp^T dz^T (per group) -> fp32 atomics.
// Causality everywhere: key j contributes to token t only when j <= t.
//
// Roles of attn_bwd_kernel (352 threads): warp 0 TMA loads of K/V, the block's work-item numbers
// and tensor-memory ownership, warp 1 the MMA issuer, warps 2 and 8-10 gather the tile's Q / dO
// rows with cp.async, warp 3 issues the dQ bulk reductions, warps 4-7 softmax / epilogue.  Tensor
// memory (512 columns): SB0, SB1 (S^T, then P^T), DB0, DB1 (dP^T, then dQ^T), dV, dK.
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tmap.h"

namespace msa {

// Row data of every query row (b, t, h), token-major: rowm[(b S + t) Hq + h] = {LSE log2 e, D}
// with D = rowsum(dO * O).
__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 c) {
  const uint32_t pa[4] = {a.x, a.y, a.z, a.w}, pc[4] = {c.x, c.y, c.z, c.w};
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&pa[e]);
    const __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162*>(&pc[e]);
    s += __low2float(x) * __low2float(y) + __high2float(x) * __high2float(y);
  }
  return s;
}

// A warp takes four consecutive rows, eight lanes per row, 32 bytes of O and of dO per lane.
__global__ void rowdot_kernel(Dims d, const bf16* __restrict__ o, const bf16* __restrict__ dout,
                              const float* __restrict__ lse, float2* __restrict__ rowm) {
  const long long rows = (long long)d.B * d.S * d.Hq;
  const int lane = threadIdx.x % 32, q = lane >> 3, l8 = lane & 7;
  const long long nw = (long long)gridDim.x * blockDim.x / 32;
  for (long long w = (blockIdx.x * (long long)blockDim.x + threadIdx.x) / 32; w * 4 < rows; w += nw) {
    const long long r = w * 4 + q;
    const bool in = r < rows;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    uint4 a0 = z, a1 = z, c0 = z, c1 = z;
    float lv = 0.f;
    if (in) {
      const uint4* po = reinterpret_cast<const uint4*>(o + (size_t)r * kD + l8 * 16);
      const uint4* pd = reinterpret_cast<const uint4*>(dout + (size_t)r * kD + l8 * 16);
      a0 = po[0];
      a1 = po[1];
      c0 = pd[0];
      c1 = pd[1];
      if (l8 == 0) {
        const int h = (int)(r % d.Hq);
        const long long bt = r / d.Hq;
        const int t = (int)(bt % d.S), b = (int)(bt / d.S);
        lv = lse[((size_t)b * d.Hq + h) * d.S + t];
      }
    }
    float s = dot8_bf16(a0, c0) + dot8_bf16(a1, c1);
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (in && l8 == 0) rowm[r] = make_float2(lv * kLog2e, s);
  }
}

namespace {
constexpr int kTR = 64;           // rows (tokens x heads) per tile
constexpr int kPG = 64;           // tokens per proxy group
constexpr int kItemTokens = 512;  // tokens per work item
constexpr int kKV = 128 * 128 * 2;  // one 128 x 128 bf16 tile (two SW128 panels)
constexpr int kRT = kTR * 128 * 2;  // one 64-row x 128 bf16 tile (two panels of 64 rows)
constexpr int kST = 128 * 128;      // dS^T / dz^T: 128 keys x 64 bf16 (one panel)
constexpr int kQS = 3;               // Q / dO slots of attn_bwd_kernel
constexpr int kSlot = 2 * kRT;         // one slot: Q rows then dO rows; later the tile's dQ staging
static_assert(kTR * 128 * 4 == kSlot, "a tile's fp32 dQ staging fills exactly one Q / dO slot");
constexpr int kIR = 4;                 // work-item ring: item numbers handed out to the block's roles

struct MainArgs {
  Dims d;
  const bf16 *q, *dout;
  const float2* emeta;  // sparse: per list entry and head, {LSE log2 e, D}
  const float2* rowm;   // dense: the same per query row [B, S, Hq] (a dense item's tokens are
                        // consecutive, so they need no per-entry copy)
  const int* seg_offset;
  const int* entries;
  const Item* items;
  const int* n_items;
  long long max_items;
  float *dq, *dk, *dv;
  __half* pbar;  // teacher rows [list entry - pass base][128 keys]: probabilities in [0, 1], fp16
  unsigned* status;
  int* sched;  // work-item counter (zero at launch): blocks take items in order as they get free
  // this pass: the items [*item_lo, *item_hi) (NULL: 0, the list's total); its teacher rows are
  // indexed from list entry *entry_lo (NULL: 0)
  const int *item_lo, *item_hi, *entry_lo;
};

struct MainShared {
  float lse2[kQS][kTR];  // row LSE * log2(e), per slot
  float drow[kQS][kTR];  // row D, per slot
  int tok[kQS][kTR];     // token position of each tile token (-1: none), per slot
  int it_ring[kIR];       // item numbers taken by this block, in order (>= total: no more)
  uint64_t kv_full, kv_empty, q_full[kQS], q_empty[kQS], stage_ready[kQS], s_full[2], p_full[2],
      ph2_full[2], s_free[2], acc_free, it_full[kIR], it_empty[kIR];
  uint32_t tmem;
};

struct ProxyArgs {
  Dims d;
  const bf16* qp;
  const float* lpxe;    // sparse: per list entry, LSE_px x log2 e
  const float* lse_px;  // dense: LSE_px per proxy row [B, Hp, S]
  const __half* pbar;  // per list entry: teacher row [128 keys] (fp16)
  float cz;          // kl_grad / (B * S * Hp), or 1 / (B * S * Hp) when czp is set
  const float* czp;  // NULL, or the device-resident kl_grad that multiplies cz
  const int* seg_offset;
  const int* entries;
  const Item* items;
  const int* n_items;
  long long max_items;
  float *dqp, *dkp;
  double* kl_acc;  // kKL: sum of pbar (ln pbar - ln p_student) over the visited pairs
  unsigned* status;
  int* sched;  // work-item counter (zero at launch)
  const int *item_lo, *item_hi, *entry_lo;  // this pass, as in MainArgs
};

constexpr int kQPB = 3;  // proxy query row buffers
constexpr int kNPB = 4;  // teacher row buffers (64 entries x 128 keys fp16 each)

struct ProxyShared {
  alignas(16) int tok[kNPB][kPG];  // per teacher buffer (read by the dz warps, 4 at a time)
  alignas(16) float lpx2[kNPB][kPG];
  int tokq[kQPB][kPG];  // per query-row buffer (read by the dQp-flush warps)
  int it_ring[kIR];  // item numbers taken by this block, in order (>= total: no more)
  uint64_t kp_full, kp_empty, qp_full[kQPB], qp_empty[kQPB], pb_full[kNPB], meta_free[kNPB], z_full[2],
      dz_full, fl_full[2], fl_free, acc_free, it_full[kIR], it_empty[kIR];
  uint32_t tmem;
};

__device__ __forceinline__ void red4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}
__device__ __forceinline__ void st_global_h_hint(__half* p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;\n" ::"l"(p),
               "h"(__half_as_ushort(__float2half_rn(v))), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void red_add_h(__half* p, float v) {
  asm volatile("red.global.add.noftz.f16 [%0], %1;\n" ::"l"(p), "h"(__half_as_ushort(__float2half_rn(v)))
               : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
// 2^x with the result flushed to zero below the normal range (probabilities that small do not
// matter here); one special-function-unit instruction.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Bulk add of `bytes` fp32 values from shared memory into global memory (TMA reduction).
__device__ __forceinline__ void bulk_reduce_add(float* g, uint32_t s, uint32_t bytes, uint64_t pol) {
  asm volatile(
      "cp.reduce.async.bulk.global.shared::cta.bulk_group.L2::cache_hint.add.f32 [%0], [%1], %2, %3;\n" ::"l"(g),
      "r"(s), "r"(bytes), "l"(pol)
      : "memory");
}
// TMA tensor reduction: adds the fp32 box staged at shared address s into the tensor at
// coordinates (c0, c1, c2); out-of-range elements of the box are skipped.
__device__ __forceinline__ void tma_reduce_add_3d(const void* tmap, int c0, int c1, int c2, uint32_t s) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], [%4];\n" ::"l"(
          tmap),
      "r"(c0), "r"(c1), "r"(c2), "r"(s)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
__device__ __forceinline__ uint32_t par(long long k) { return (uint32_t)(k & 1); }

// First token of a dense item / first entry of a sparse item.
template <bool kDense>
__device__ __forceinline__ long long item_base(const Dims& d, const int* seg_offset, const Item& it) {
  if (kDense) {
    const long long n = it.seg % d.nblk, c = it.seg / d.nseg();
    const long long lo = (long long)c * d.chunk;
    return (n * kBlock > lo ? n * kBlock : lo) + it.first;
  }
  return (long long)seg_offset[it.seg] + it.first;
}
}  // namespace

// ==========================================================================================
template <int G, bool kDense>
__global__ void __launch_bounds__(352, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    MainArgs A) {
  using namespace sm100;
  constexpr int TT = kTR / G;  // tokens per tile
  // With 16 heads per group, up to 16 x (tokens) rows add into each key's dV and dK; P and dS
  // rounded once to bf16 for dV = P^T dO and dK = dS^T Q then cost up to ~2e-2 on the largest
  // entries.  So P^T is written as its bf16 value plus the bf16 residual P - bf16(P) (columns 32-63
  // of the same buffer), dS^T's residual goes to the dP^T buffer (its columns are read just before,
  // and dQ^T overwrites them only after the dK products, in issue order), and dV, dK take both
  // parts (to ~16 significant bits; eight more MMAs a tile).
  constexpr bool kSplitP = G >= 16;
  const Dims& d = A.d;

  extern __shared__ uint8_t smem_raw[];
  MainShared* sh = reinterpret_cast<MainShared*>(smem_raw);
  uint8_t* base = align1024(smem_raw + sizeof(MainShared));
  uint8_t* sK = base;                  // [128 keys][128 d]  (TMA)
  uint8_t* sV = sK + kKV;
  uint8_t* sSl = sV + kKV;             // [kQS] slots: Q [64 rows][128 d], dO [64 rows][128 d]
  uint8_t* sdS = sSl + kQS * kSlot;    // [2] dS^T [128 keys][64 rows]
  const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aSl = smem_u32(sSl), adS = smem_u32(sdS);

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const float sl2 = d.scale * kLog2e;
  long long total = A.item_hi ? *A.item_hi : *A.n_items;  // items of this pass end here
  if (total > A.max_items) total = A.max_items;
  const int item0 = A.item_lo ? *A.item_lo : 0;
  const long long ent0 = A.entry_lo ? *A.entry_lo : 0;  // list entry of teacher row 0

  if (tid == 0) {
    mbar_init(&sh->kv_full, 1);
    mbar_init(&sh->kv_empty, 1);
    for (int x = 0; x < kQS; ++x) {
      mbar_init(&sh->q_full[x], 256);  // 4 gather warps x 32 lanes: a cp.async and a plain arrival each
      mbar_init(&sh->q_empty[x], 1);   // the dQ reducer, once the staged dQ rows were read
      mbar_init(&sh->stage_ready[x], 4);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sh->s_full[x], 1);
      mbar_init(&sh->p_full[x], 4);
      mbar_init(&sh->ph2_full[x], 1);
      mbar_init(&sh->s_free[x], 4);
    }
    mbar_init(&sh->acc_free, 4);
    for (int x = 0; x < kIR; ++x) {
      mbar_init(&sh->it_full[x], 1);
      mbar_init(&sh->it_empty[x], 10);  // MMA, 4 gather warps, reducer, 4 softmax warps
    }
    mbar_fence_init();
  }
  if (warp == 0) {
    __syncwarp();  // lane 0 initialised the barriers alone; the allocation is warp-collective
    tmem_alloc(&sh->tmem, 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sh->tmem;
  const uint32_t SB0 = tmem, DB0 = tmem + 128, RV = tmem + 256, RK = tmem + 384;
  bool ok = true;
  // Item number ni of this block, for one thread / for a whole warp.  Items are handed out in list
  // order to whichever block asks next, so the blocks stay within a short window of the list (the
  // rows of one sequence chunk stay in L2) however unevenly long the items are.
  auto take_item1 = [&](long long ni, int& v) -> bool {
    const int x = (int)(ni % kIR);
    if (!mbar_wait(&sh->it_full[x], par(ni / kIR), A.status)) return false;
    v = sh->it_ring[x];
    mbar_arrive(&sh->it_empty[x]);
    return true;
  };
  auto take_itemw = [&](long long ni, int& v) -> bool {
    const int x = (int)(ni % kIR);
    if (!mbar_wait_warp(&sh->it_full[x], par(ni / kIR), A.status)) return false;
    v = sh->it_ring[x];
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh->it_empty[x]);
    return true;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA: K, V per item
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      // item numbers are published up to two items ahead of the K / V loads
      long long pub = 0;
      bool last = false;
      for (long long ni = 0;; ++ni) {
        while (!last && pub < ni + 2) {
          const int x = (int)(pub % kIR);
          if (pub >= kIR && !mbar_wait(&sh->it_empty[x], par(pub / kIR - 1), A.status)) break;
          const int v = item0 + atomicAdd(A.sched, 1);
          sh->it_ring[x] = v;
          mbar_arrive(&sh->it_full[x]);
          last = v >= total;
          ++pub;
        }
        if (pub <= ni) break;  // a wait gave up
        const int it = sh->it_ring[ni % kIR];
        if (it >= total) break;
        const Item item = A.items[it];
        const int n = item.seg % d.nblk;
        const int bg = (int)((item.seg % d.nseg()) / d.nblk);
        const int b = bg / d.Hp, kvh = d.kv_of((bg % d.Hp) * d.R + item.sub);
        if (ni > 0 && !mbar_wait(&sh->kv_empty, par(ni - 1), A.status)) break;
        const int row0 = b * d.S + n * kBlock;
        mbar_expect_tx(&sh->kv_full, 2 * kKV);
        tma_load_3d(sK, &tm_k, 0, kvh, row0, &sh->kv_full);
        tma_load_3d(sK + kKV / 2, &tm_k, 64, kvh, row0, &sh->kv_full);
        tma_load_3d(sV, &tm_v, 0, kvh, row0, &sh->kv_full);
        tma_load_3d(sV + kKV / 2, &tm_v, 64, kvh, row0, &sh->kv_full);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, kTR, false, false);  // S^T, dP^T
      constexpr uint32_t id_g = idesc_bf16(128, 128, false, true);   // dV, dK
      constexpr uint32_t id_q = idesc_bf16(128, kTR, true, true);    // dQ^T
      long long ni = 0, i = 0;
      bool first_of_item = true;
      auto phase2 = [&](long long ti) -> bool {
        const int b = (int)(ti & 1);
        if (!mbar_wait(&sh->p_full[b], par(ti >> 1), A.status)) return false;
        if (first_of_item && ni > 0 && !mbar_wait(&sh->acc_free, par(ni - 1), A.status)) return false;
        fence_after_sync();
        const bool acc = !first_of_item;
        first_of_item = false;
        const uint32_t aQb = aSl + (uint32_t)(ti % kQS) * kSlot, adOb = aQb + kRT, adSb = adS + b * kST;
        const uint32_t SBb = SB0 + 64 * b, DBb = DB0 + 64 * b;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // dV += P^T dO  (P^T from tensor memory)
          mma_ts(RV, SBb + ks * 8, desc_mnmajor(adOb, kTR, ks), id_g, acc || ks > 0);
        if constexpr (kSplitP) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)  // dV += P_lo^T dO  (the bf16 residual of P)
            mma_ts(RV, SBb + 32 + ks * 8, desc_mnmajor(adOb, kTR, ks), id_g, true);
        }
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // dK += dS^T Q
          mma_ss(RK, desc_kmajor(adSb, 128, ks), desc_mnmajor(aQb, kTR, ks), id_g, acc || ks > 0);
        if constexpr (kSplitP) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)  // dK += dS_lo^T Q  (the bf16 residual, from DB_b)
            mma_ts(RK, DBb + ks * 8, desc_mnmajor(aQb, kTR, ks), id_g, true);
        }
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)  // dQ^T = K^T dS^T
          mma_ss(DBb, desc_mnmajor(aK, 128, ks), desc_mnmajor(adSb, 128, ks), id_q, ks > 0);
        mma_commit(&sh->ph2_full[b]);  // also: the slot's Q / dO rows are no longer read
        return true;
      };
      for (;; ++ni) {
        int it;
        if (!take_item1(ni, it)) { ok = false; break; }
        if (it >= total) break;
        const Item item = A.items[it];
        if (!mbar_wait(&sh->kv_full, par(ni), A.status)) { ok = false; break; }
        first_of_item = true;
        const int ntiles = (item.count + TT - 1) / TT;
        for (int tl = 0; tl < ntiles; ++tl, ++i) {
          const int b = (int)(i & 1), sl = (int)(i % kQS);
          if (!mbar_wait(&sh->q_full[sl], par(i / kQS), A.status)) { ok = false; break; }
          // the Q / dO rows were written by other threads' cp.async (generic proxy) and are only
          // tracked by the barrier: order them before the tensor core's (async proxy) reads
          fence_async_smem();
          fence_after_sync();
          const uint32_t aQb = aSl + (uint32_t)sl * kSlot, adOb = aQb + kRT;
          // SB_b last held P^T of tile i-2, read by that tile's phase 2, issued earlier
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // S^T = K Q^T
            mma_ss(SB0 + 64 * b, desc_kmajor(aK, 128, ks), desc_kmajor(aQb, kTR, ks), id_s, ks > 0);
          // DB_b holds dQ^T of tile i-2 until the epilogue has read it out
          if (i >= 2 && !mbar_wait(&sh->s_free[b], par((i - 2) >> 1), A.status)) { ok = false; break; }
          fence_after_sync();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // dP^T = V dO^T
            mma_ss(DB0 + 64 * b, desc_kmajor(aV, 128, ks), desc_kmajor(adOb, kTR, ks), id_s, ks > 0);
          mma_commit(&sh->s_full[b]);
          if (tl > 0 && !phase2(i - 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (!phase2(i - 1)) { ok = false; break; }
        mma_commit(&sh->kv_empty);
      }
    }
  } else if (warp == 2 || warp >= 8) {
    // ---------------------------------------------------------------- gather: Q, dO rows
    // Four warps (2, 8, 9, 10) each fill 16 of the tile's 64 rows with cp.async; completion is
    // counted on q_full (one cp.async arrival and one plain arrival per lane), so a warp moves on
    // to the next tile as soon as its copies are issued.  (Q rows as per-token TMA boxes were
    // slower: the TMA unit also carries the dQ bulk reductions.)
    const uint64_t keep = l2_policy_evict_last();  // read again by the chunk's other blocks
    const int gw = warp == 2 ? 0 : warp - 7;
    constexpr int WT = 16 / G;  // tokens of one warp's 16 rows (G in {4, 8, 16})
    const int r0 = 16 * gw;
    const int hi = lane >> 4, ch = lane & 15;
    long long i = 0;
    for (long long ni = 0; ok; ++ni) {
      int it;
      if (!take_itemw(ni, it)) { ok = false; break; }
      if (it >= total) break;
      const Item item = A.items[it];
      const int bg = (int)((item.seg % d.nseg()) / d.nblk);
      const int b = bg / d.Hp, a = (bg % d.Hp) * d.R + item.sub;  // attention group
      const int gp = d.Gp();  // row data per entry: the proxy head's Gp query heads
      const long long tb = item_base<kDense>(d, A.seg_offset, item);
      const long long eb = (long long)A.seg_offset[item.seg] + item.first;  // first list entry
      auto load_tokens = [&](int pos0, int valid, int (&tv)[TT]) {
#pragma unroll
        for (int x = 0; x < TT; ++x)
          tv[x] = x < valid ? (kDense ? (int)(tb + pos0 + x) : (__ldg(A.entries + tb + pos0 + x) >> 8)) : -1;
      };
      // row data of row r0 + (lane & 15) of tile tl_ (lanes 0-15), indexed by the list entry
      // (dense: by the token, tb + x), so it needs no token first
      auto load_meta = [&](int tl_) -> float2 {
        const int x = tl_ * TT + (r0 + ch) / G;
        const int h = item.sub * G + (r0 + ch) % G;  // query head within the proxy head's Gp
        float2 m = make_float2(0.f, 0.f);
        if (hi == 0 && x < item.count)
          m = kDense ? __ldg(A.rowm + ((size_t)b * d.S + tb + x) * d.Hq + (size_t)(bg % d.Hp) * gp + h)
                     : __ldg(A.emeta + (size_t)(eb + x) * gp + h);
        return m;
      };
      const int ntiles = (item.count + TT - 1) / TT;
      int tv[TT];
      load_tokens(0, min(TT, item.count), tv);
      float2 mcur = load_meta(0);
      for (int tl = 0; tl < ntiles; ++tl, ++i) {
        const int sl = (int)(i % kQS);
        int wt[WT];  // this warp's tokens
#pragma unroll
        for (int j = 0; j < WT; ++j) {
          wt[j] = -1;
#pragma unroll
          for (int x = 0; x < TT; ++x)
            if (x == r0 / G + j) wt[j] = tv[x];
        }
        const int mr = r0 + ch;
        int tn[TT];
        load_tokens((tl + 1) * TT, min(TT, item.count - (tl + 1) * TT), tn);
        const float2 mnext = load_meta(tl + 1);
        if (i >= kQS && !mbar_wait_warp(&sh->q_empty[sl], par(i / kQS - 1), A.status)) { ok = false; break; }
        uint8_t* dQb = sSl + sl * kSlot;
        uint8_t* ddOb = dQb + kRT;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int rr = 2 * k + hi;  // row within the warp's 16
          const int r = r0 + rr;
          const int t = wt[(2 * k) / G];
          const uint32_t off = (ch >> 3) * (kTR * 128) + sm100::sw128_chunk(r, ch & 7);
          const size_t grow = (((size_t)b * d.S + (t < 0 ? 0 : t)) * d.Hq + a * G + rr % G) * kD + ch * 8;
          cp_async16_hint(dQb + off, A.q + grow, t >= 0, keep);
          cp_async16_hint(ddOb + off, A.dout + grow, t >= 0, keep);
        }
        if (hi == 0) {
          sh->lse2[sl][mr] = mcur.x;
          sh->drow[sl][mr] = mcur.y;
        }
        if (gw == 0) {
#pragma unroll
          for (int x = 0; x < TT; ++x)
            if (lane == x) sh->tok[sl][x] = tv[x];
        }
        cp_async_arrive(&sh->q_full[sl]);
        mbar_arrive(&sh->q_full[sl]);  // publishes the row data and tok
#pragma unroll
        for (int x = 0; x < TT; ++x) tv[x] = tn[x];
        mcur = mnext;
      }
    }
    cp_async_wait_all();  // nothing may land after the block exits
  } else if (warp == 3) {
    // ---------------------------------------------------------------- dQ reducer
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();  // dQ rows of the chunk: reduced into again
      long long ns = 0;
      for (long long ni = 0; ok; ++ni) {
        int it;
        if (!take_item1(ni, it)) { ok = false; break; }
        if (it >= total) break;
        const Item item = A.items[it];
        const int bg = (int)((item.seg % d.nseg()) / d.nblk);
        const int b = bg / d.Hp, a = (bg % d.Hp) * d.R + item.sub;  // attention group
        const int ntiles = (item.count + TT - 1) / TT;
        for (int tl = 0; tl < ntiles; ++tl, ++ns) {
          const int sl = (int)(ns % kQS);
          if (!mbar_wait(&sh->stage_ready[sl], par(ns / kQS), A.status)) { ok = false; break; }
          const uint32_t aSt = aSl + (uint32_t)sl * kSlot;  // the tile's dQ rows, staged in its slot
#pragma unroll 1
          for (int x = 0; x < TT; ++x) {
            const int t = sh->tok[sl][x];
            if (t >= 0)
              bulk_reduce_add(A.dq + (((size_t)b * d.S + t) * d.Hq + a * G) * kD,
                              aSt + x * G * kD * 4, G * kD * 4, keep);
          }
          bulk_commit();
          bulk_wait_read0();
          mbar_arrive(&sh->q_empty[sl]);  // the slot may take the rows of tile ns + kQS
        }
      }
      bulk_wait0();
    }
  } else {
    // ---------------------------------------------------------------- softmax / epilogue
    const int w4 = warp - 4;
    const int kr = w4 * 32 + lane;  // key row of S^T / dP^T (TMEM lane); head-dim index of dQ^T
    const uint32_t lb = static_cast<uint32_t>(w4 * 32) << 16;
    const uint64_t stream = l2_policy_evict_first();  // pbar rows: read once, by proxy_bwd
    long long i = 0;
    // dQ of tile ti: dQ^T (tensor memory) -> fp32 rows staged in the tile's own slot, whose Q / dO
    // rows phase 2 has finished reading; the reducer warp then adds them to dQ
    auto epilogue = [&](long long ti) -> bool {
      const int bb = (int)(ti & 1), sl = (int)(ti % kQS);
      __syncwarp();
      if (!mbar_wait_warp(&sh->ph2_full[bb], par(ti >> 1), A.status)) return false;
      fence_after_sync();
      float* stage = reinterpret_cast<float*>(sSl + sl * kSlot);
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t r0[32];
        __syncwarp();
        tmem_ld32(DB0 + 64 * bb + lb + 32 * c, r0);
        tmem_wait_ld();
#pragma unroll
        for (int r = 0; r < 32; ++r) stage[(32 * c + r) * kD + kr] = __uint_as_float(r0[r]) * d.scale;
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->s_free[bb]);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->stage_ready[sl]);
      return true;
    };
    for (long long ni = 0; ok; ++ni) {
      int it;
      if (!take_itemw(ni, it)) { ok = false; break; }
      if (it >= total) break;
      const Item item = A.items[it];
      const int n = item.seg % d.nblk;
      const int bg = (int)((item.seg % d.nseg()) / d.nblk);
      const int b = bg / d.Hp, kvh = d.kv_of((bg % d.Hp) * d.R + item.sub);
      const int j = n * kBlock + kr;  // this thread's key
      const long long eb = (long long)A.seg_offset[item.seg] + item.first;  // first list entry
      const int ntiles = (item.count + TT - 1) / TT;
      for (int tl = 0; tl < ntiles; ++tl, ++i) {
        const int bb = (int)(i & 1), sl = (int)(i % kQS);
        __syncwarp();
        if (!mbar_wait_warp(&sh->q_full[sl], par(i / kQS), A.status) ||
            !mbar_wait_warp(&sh->s_full[bb], par(i >> 1), A.status)) {
          ok = false;
          break;
        }
        fence_after_sync();
        // ---- softmax of tile i
        int tv[TT];
        bool vis[TT];
        float pb[TT];
#pragma unroll
        for (int x = 0; x < TT; ++x) {
          tv[x] = sh->tok[sl][x];
          vis[x] = tv[x] >= 0 && j <= tv[x];
          pb[x] = 0.f;
        }
        const uint32_t SBb = SB0 + 64 * bb, DBb = DB0 + 64 * bb;
        const uint32_t adSb = adS + bb * kST;
        // kSplitP: the bf16 residual P - bf16(P) of rows 0-31, written to columns 32-47 only once
        // the S^T values of rows 32-63 in those columns have been read
        uint32_t lw0[kSplitP ? 16 : 1];
#pragma unroll
        for (int c = 0; c < 2; ++c) {  // 32 rows at a time (P^T of rows 0-31 lands in columns 0-15)
          uint32_t rs[32], rp[32];
          __syncwarp();
          tmem_ld32(SBb + lb + 32 * c, rs);
          tmem_ld32(DBb + lb + 32 * c, rp);
          tmem_wait_ld();
          uint32_t pw[16], dw[16];
          uint32_t lw[kSplitP ? 16 : 1], dlw[kSplitP ? 16 : 1];
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const float4 l4 = reinterpret_cast<const float4*>(sh->lse2[sl])[c * 8 + q4];
            const float4 d4 = reinterpret_cast<const float4*>(sh->drow[sl])[c * 8 + q4];
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
            const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
            float pv[4], dsv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int r = c * 32 + q4 * 4 + e;
              const int x = r / G;
              const float sv = __uint_as_float(rs[q4 * 4 + e]);
              const float dpv = __uint_as_float(rp[q4 * 4 + e]);
              const float p = vis[x] ? ex2(sv * sl2 - lv[e]) : 0.f;
              pv[e] = p;
              dsv[e] = p * (dpv - dv4[e]);
              pb[x] += p;
            }
            pw[2 * q4] = pack_bf16(pv[0], pv[1]);
            pw[2 * q4 + 1] = pack_bf16(pv[2], pv[3]);
            dw[2 * q4] = pack_bf16(dsv[0], dsv[1]);
            dw[2 * q4 + 1] = pack_bf16(dsv[2], dsv[3]);
            if constexpr (kSplitP) {
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&pw[2 * q4 + h2]);
                lw[2 * q4 + h2] = pack_bf16(pv[2 * h2] - __low2float(hi), pv[2 * h2 + 1] - __high2float(hi));
                const __nv_bfloat162 dh = *reinterpret_cast<const __nv_bfloat162*>(&dw[2 * q4 + h2]);
                dlw[2 * q4 + h2] = pack_bf16(dsv[2 * h2] - __low2float(dh), dsv[2 * h2 + 1] - __high2float(dh));
              }
            }
          }
          tmem_st16(SBb + lb + c * 16, pw);  // P^T: row r packed into column r / 2
          if constexpr (kSplitP) {
            // dS^T residual of these 32 rows over dP^T columns 16 c .. 16 c + 15, already read
            tmem_st16(DBb + lb + c * 16, dlw);
            if (c == 0) {
#pragma unroll
              for (int u = 0; u < 16; ++u) lw0[u] = lw[u];
            } else {  // every S^T column of this warp's lanes has been read: residuals to 32-63
              tmem_st16(SBb + lb + 32, lw0);
              tmem_st16(SBb + lb + 48, lw);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
            st_shared_v4(adSb + sm100::sw128_chunk(kr, c * 4 + u), dw[4 * u], dw[4 * u + 1],
                         dw[4 * u + 2], dw[4 * u + 3]);
        }
        tmem_wait_st();
        fence_async_smem();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->p_full[bb]);
        // teacher: mean of the proxy head's G R query heads' probabilities of each token, one fp16
        // row per list entry; with R > 1 attention groups per proxy head each adds its share
        if (d.R == 1) {
#pragma unroll
          for (int x = 0; x < TT; ++x)
            if (tv[x] >= 0)
              st_global_h_hint(A.pbar + (size_t)(eb - ent0 + tl * TT + x) * kBlock + kr, pb[x] * (1.f / G), stream);
        } else {
#pragma unroll
          for (int x = 0; x < TT; ++x)
            if (tv[x] >= 0)
              red_add_h(A.pbar + (size_t)(eb - ent0 + tl * TT + x) * kBlock + kr, pb[x] * (1.f / (G * d.R)));
        }
        // ---- epilogue of the previous tile
        if (tl > 0 && !epilogue(i - 1)) { ok = false; break; }
      }
      if (!ok) break;
      if (!epilogue(i - 1)) { ok = false; break; }
      // ---- item end: dV and dK rows of this key
      {
        float* pv = A.dv + (((size_t)b * d.S + j) * d.Hkv + kvh) * kD;
        float* pk = A.dk + (((size_t)b * d.S + j) * d.Hkv + kvh) * kD;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t rv[32], rk[32];
          tmem_ld32(RV + lb + c * 32, rv);
          tmem_ld32(RK + lb + c * 32, rk);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            red4(pv + c * 32 + 4 * u, __uint_as_float(rv[4 * u]), __uint_as_float(rv[4 * u + 1]),
                 __uint_as_float(rv[4 * u + 2]), __uint_as_float(rv[4 * u + 3]));
            red4(pk + c * 32 + 4 * u, __uint_as_float(rk[4 * u]) * d.scale,
                 __uint_as_float(rk[4 * u + 1]) * d.scale, __uint_as_float(rk[4 * u + 2]) * d.scale,
                 __uint_as_float(rk[4 * u + 3]) * d.scale);
          }
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->acc_free);
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ==========================================================================================
// The same backward with 128-row tiles (128 / G tokens x G heads): every product then has N = 128,
// which the tensor core runs in the time of an N = 64 one -- 40 MMA instructions per 128 rows
// instead of 64 with two 64-row tiles.  Tensor memory holds one tile's S^T (then P^T) and dP^T
// (then dS^T, then dQ^T) besides dV and dK, so the S / dP products of a tile wait for the previous tile's
// epilogue instead of running ahead of it; the tensor core idles while the softmax runs.  To keep
// that gap short the softmax and epilogue of a tile are split over eight warps: two per
// tensor-memory lane quarter, one for the tile's rows 0-63 and one for rows 64-127.  Shared memory
// (1024-aligned base): K, V (32 KB each), two Q / dO slots of 64 KB (each later holding its tile's
// fp32 dQ rows), dS^T (32 KB) and the barriers -- 224 KB + the barrier block.
// Roles (16 warps): 0 TMA of K / V, 1 MMA issue, 3 dQ reducer, 4-11 softmax / epilogue, 12-15
// gather of the Q / dO rows; warp 2 has no role.
namespace {
constexpr int kTW = 128;             // rows per wide tile
constexpr int kRTW = kTW * 128 * 2;  // 128 rows x 128 bf16 (two SW128 panels of 64 columns)
constexpr int kSlotW = 2 * kRTW;     // Q rows, then dO rows; later the tile's fp32 dQ rows
constexpr int kSTW = 128 * kTW * 2;  // dS^T: 128 keys x 128 rows bf16 (two panels)
constexpr int kQSW = 2;              // Q / dO slots
constexpr int kWideThreads = 512;    // 16 warps
constexpr int kSoftW = 8;            // softmax / epilogue warps
static_assert(kTW * 128 * 4 == kSlotW, "a wide tile's fp32 dQ staging fills exactly one slot");
constexpr uint32_t kStatusLayout = kStatusInternal;  // dynamic shared memory not 1024-byte aligned

struct WideShared {
  float nlse2[kQSW][kTW];  // -(row LSE * log2(e)), per slot
  float ndrow[kQSW][kTW];  // -(row D) * scale, per slot
  int tok[kQSW][32];      // tokens of the slot's tile (128 / G <= 32), -1: none
  int it_ring[kIR];
  uint64_t kv_full, kv_empty, q_full[kQSW], q_empty[kQSW], stage_ready[kQSW], s_full, p_full,
      ph2_full, s_free, acc_free, mma_done, it_full[kIR], it_empty[kIR];
  uint32_t tmem;
};
constexpr size_t kWideSmem = 2 * (size_t)kKV + kQSW * (size_t)kSlotW + kSTW;  // + WideShared
}  // namespace

template <int G, bool kDense>
__global__ void __launch_bounds__(kWideThreads, 1)
    attn_bwd_wide_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         MainArgs A) {
  using namespace sm100;
  constexpr int TT = kTW / G;  // tokens per tile
  static_assert(TT <= 32 && G >= 4, "one lane per token of a tile");
  const Dims& d = A.d;
  extern __shared__ __align__(1024) uint8_t smem_wide[];
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  if (smem_u32(smem_wide) & 1023u) {  // the swizzled operand layout needs 1024-byte atoms
    if (tid == 0) atomicOr(A.status, kStatusLayout);
    return;
  }
  uint8_t* sK = smem_wide;  // [128 keys][128 d]  (TMA)
  uint8_t* sV = sK + kKV;
  uint8_t* sSl = sV + kKV;              // [kQSW] slots: Q [128 rows][128 d], dO [128 rows][128 d]
  uint8_t* sdS = sSl + kQSW * kSlotW;   // dS^T [128 keys][128 rows]
  WideShared* sh = reinterpret_cast<WideShared*>(sdS + kSTW);
  const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aSl = smem_u32(sSl), adS = smem_u32(sdS);
  const float sl2 = d.scale * kLog2e;
  long long total = A.item_hi ? *A.item_hi : *A.n_items;  // items of this pass end here
  if (total > A.max_items) total = A.max_items;
  const int item0 = A.item_lo ? *A.item_lo : 0;
  const long long ent0 = A.entry_lo ? *A.entry_lo : 0;  // list entry of teacher row 0

  if (tid == 0) {
    mbar_init(&sh->kv_full, 1);
    mbar_init(&sh->kv_empty, 1);
    for (int x = 0; x < kQSW; ++x) {
      mbar_init(&sh->q_full[x], 256);  // 4 gather warps x 32 lanes: a cp.async and a plain arrival each
      mbar_init(&sh->q_empty[x], 1);   // the dQ reducer, once the staged dQ rows were read
      mbar_init(&sh->stage_ready[x], kSoftW);
    }
    mbar_init(&sh->s_full, 1);
    mbar_init(&sh->p_full, kSoftW);
    mbar_init(&sh->ph2_full, 1);
    mbar_init(&sh->s_free, kSoftW);
    mbar_init(&sh->acc_free, kSoftW);
    mbar_init(&sh->mma_done, 1);
    for (int x = 0; x < kIR; ++x) {
      mbar_init(&sh->it_full[x], 1);
      mbar_init(&sh->it_empty[x], 6 + kSoftW);  // MMA, 4 gather warps, reducer, softmax warps
    }
    mbar_fence_init();
  }
  if (warp == 0) {
    __syncwarp();  // lane 0 initialised the barriers alone; the allocation is warp-collective
    tmem_alloc(&sh->tmem, 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sh->tmem;
  const uint32_t SB = tmem, DB = tmem + 128, RV = tmem + 256, RK = tmem + 384;
  bool ok = true;
  // waits record which of them gave up first (status word kStatusWhere), so that a deadlock is
  // reported with its place instead of leaving only the timeout bit
  auto wait1 = [&](unsigned id, uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_wait(bar, parity, A.status)) return true;
    atomicCAS(A.status + kStatusWhere, 0u, id);
    return false;
  };
  auto waitw = [&](unsigned id, uint64_t* bar, uint32_t parity) -> bool {
    const bool r = wait1(id, bar, parity);
    return __all_sync(0xffffffffu, r);
  };
  auto take_item1 = [&](long long ni, int& v) -> bool {
    const int x = (int)(ni % kIR);
    if (!wait1(1, &sh->it_full[x], par(ni / kIR))) return false;
    v = sh->it_ring[x];
    mbar_arrive(&sh->it_empty[x]);
    return true;
  };
  auto take_itemw = [&](long long ni, int& v) -> bool {
    const int x = (int)(ni % kIR);
    if (!waitw(2, &sh->it_full[x], par(ni / kIR))) return false;
    v = sh->it_ring[x];
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh->it_empty[x]);
    return true;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA: K, V per item
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      long long pub = 0;
      bool last = false;
      for (long long ni = 0;; ++ni) {
        while (!last && pub < ni + 2) {  // item numbers up to two items ahead of the loads
          const int x = (int)(pub % kIR);
          if (pub >= kIR && !wait1(3, &sh->it_empty[x], par(pub / kIR - 1))) break;
          const int v = item0 + atomicAdd(A.sched, 1);
          sh->it_ring[x] = v;
          mbar_arrive(&sh->it_full[x]);
          last = v >= total;
          ++pub;
        }
        if (pub <= ni) break;  // a wait gave up
        const int it = sh->it_ring[ni % kIR];
        if (it >= total) break;
        const Item item = A.items[it];
        const int n = item.seg % d.nblk;
        const int bg = (int)((item.seg % d.nseg()) / d.nblk);
        const int b = bg / d.Hp, kvh = d.kv_of((bg % d.Hp) * d.R + item.sub);
        if (ni > 0 && !wait1(4, &sh->kv_empty, par(ni - 1))) break;
        const int row0 = b * d.S + n * kBlock;
        mbar_expect_tx(&sh->kv_full, 2 * kKV);
        tma_load_3d(sK, &tm_k, 0, kvh, row0, &sh->kv_full);
        tma_load_3d(sK + kKV / 2, &tm_k, 64, kvh, row0, &sh->kv_full);
        tma_load_3d(sV, &tm_v, 0, kvh, row0, &sh->kv_full);
        tma_load_3d(sV + kKV / 2, &tm_v, 64, kvh, row0, &sh->kv_full);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, kTW, false, false);  // S^T, dP^T (N = rows)
      constexpr uint32_t id_g = idesc_bf16(128, 128, false, true);   // dV, dK (N = d)
      constexpr uint32_t id_q = idesc_bf16(128, kTW, true, true);    // dQ^T (N = rows)
      long long i = 0;
      for (long long ni = 0;; ++ni) {
        int it;
        if (!take_item1(ni, it)) { ok = false; break; }
        if (it >= total) break;
        const Item item = A.items[it];
        if (!wait1(5, &sh->kv_full, par(ni))) { ok = false; break; }
        const int ntiles = (item.count + TT - 1) / TT;
        for (int tl = 0; tl < ntiles; ++tl, ++i) {
          const int sl = (int)(i % kQSW);
          if (!wait1(6, &sh->q_full[sl], par(i / kQSW))) { ok = false; break; }
          // the Q / dO rows came from other threads' cp.async (generic proxy), tracked by q_full
          fence_async_smem();
          fence_after_sync();
          const uint32_t aQb = aSl + (uint32_t)sl * kSlotW, adOb = aQb + kRTW;
          // S^T = K Q^T into SB, which held P^T of tile i-1 (read by that tile's dV product,
          // issued before this one)
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ss(SB, desc_kmajor(aK, 128, ks), desc_kmajor(aQb, kTW, ks), id_s, ks > 0);
          // dP^T = V dO^T into DB, once the epilogue of tile i-1 has read dQ^T out of it
          if (i >= 1 && !wait1(7, &sh->s_free, par(i - 1))) { ok = false; break; }
          fence_after_sync();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ss(DB, desc_kmajor(aV, 128, ks), desc_kmajor(adOb, kTW, ks), id_s, ks > 0);
          mma_commit(&sh->s_full);  // also: every product of tile i-1 has completed
          // phase 2, once the softmax has written P^T (tensor memory) and dS^T (tensor memory for
          // dK, shared memory for dQ^T)
          if (!wait1(8, &sh->p_full, par(i))) { ok = false; break; }
          if (tl == 0 && ni > 0 && !wait1(9, &sh->acc_free, par(ni - 1))) { ok = false; break; }
          fence_after_sync();
          const bool acc = tl > 0;
          // dK += dS^T Q and dV += P^T dO with dS^T and P^T read from tensor memory (rows 0-63 in
          // columns 0-31 of DB / SB, rows 64-127 in columns 64-95), which spares the shared-memory
          // path a 32 KB operand per tile; dK first, so that the dV products separate its reads
          // of DB from the dQ^T product that overwrites DB
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ts(RK, DB + ks * 8 + (ks >= 4 ? 32 : 0), desc_mnmajor(aQb, kTW, ks), id_g,
                   acc || ks > 0);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ts(RV, SB + ks * 8 + (ks >= 4 ? 32 : 0), desc_mnmajor(adOb, kTW, ks), id_g,
                   acc || ks > 0);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // dQ^T = K^T dS^T into DB (B operand: dS^T in shared memory)
            mma_ss(DB, desc_mnmajor(aK, 128, ks), desc_mnmajor(adS, 128, ks), id_q, ks > 0);
          mma_commit(&sh->ph2_full);  // also: the slot's Q / dO rows are no longer read
        }
        if (!ok) break;
        mma_commit(&sh->kv_empty);
      }
      mma_commit(&sh->mma_done);  // arrives once every MMA issued above has completed
    }
  } else if (warp >= 12) {
    // ---------------------------------------------------------------- gather: Q, dO rows
    // Four warps (12-15) each fill 32 of the tile's 128 rows with cp.async; completion is counted
    // on q_full (one cp.async arrival and one plain arrival per lane).  Lane x holds token x of the
    // tile (one tile ahead); warp 12 publishes them for the reducer and the softmax.
    const uint64_t keep = l2_policy_evict_last();  // read again by the chunk's other blocks
    const int gw = warp - 12;
    constexpr int WT = 32 / G;  // tokens of one warp's 32 rows
    const int r0 = 32 * gw;
    const int hi = lane >> 4, ch = lane & 15;
    long long i = 0;
    for (long long ni = 0; ok; ++ni) {
      int it;
      if (!take_itemw(ni, it)) { ok = false; break; }
      if (it >= total) break;
      const Item item = A.items[it];
      const int bg = (int)((item.seg % d.nseg()) / d.nblk);
      const int b = bg / d.Hp, a = (bg % d.Hp) * d.R + item.sub;  // attention group
      const int gp = d.Gp();
      const long long tb = item_base<kDense>(d, A.seg_offset, item);
      const long long eb = (long long)A.seg_offset[item.seg] + item.first;  // first list entry
      // token of tile position `lane` of tile tl_ (-1: none)
      auto load_tok = [&](int tl_) -> int {
        const int x = tl_ * TT + lane;
        if (lane >= TT || x >= item.count) return -1;
        return kDense ? (int)(tb + x) : (__ldg(A.entries + tb + x) >> 8);
      };
      // row data of row r0 + lane of tile tl_, indexed by the list entry (dense: by the token)
      auto load_meta = [&](int tl_) -> float2 {
        const int x = tl_ * TT + (r0 + lane) / G;
        const int h = item.sub * G + (r0 + lane) % G;  // query head within the proxy head's Gp
        float2 m = make_float2(0.f, 0.f);
        if (x < item.count)
          m = kDense ? __ldg(A.rowm + ((size_t)b * d.S + tb + x) * d.Hq + (size_t)(bg % d.Hp) * gp + h)
                     : __ldg(A.emeta + (size_t)(eb + x) * gp + h);
        return m;
      };
      const int ntiles = (item.count + TT - 1) / TT;
      int tcur = load_tok(0);
      float2 mcur = load_meta(0);
      for (int tl = 0; tl < ntiles; ++tl, ++i) {
        const int sl = (int)(i % kQSW);
        int wt[WT];  // this warp's tokens
#pragma unroll
        for (int j = 0; j < WT; ++j) wt[j] = __shfl_sync(0xffffffffu, tcur, r0 / G + j);
        const int tnext = load_tok(tl + 1);
        const float2 mnext = load_meta(tl + 1);
        if (i >= kQSW && !waitw(10, &sh->q_empty[sl], par(i / kQSW - 1))) { ok = false; break; }
        uint8_t* dQb = sSl + sl * kSlotW;
        uint8_t* ddOb = dQb + kRTW;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int rr = 2 * k + hi;  // row within the warp's 32 (G >= 4: token (2 k) / G)
          const int r = r0 + rr;
          const int t = wt[(2 * k) / G];
          const uint32_t off = (ch >> 3) * (kTW * 128) + sm100::sw128_chunk(r, ch & 7);
          const size_t grow = (((size_t)b * d.S + (t < 0 ? 0 : t)) * d.Hq + a * G + rr % G) * kD + ch * 8;
          cp_async16_hint(dQb + off, A.q + grow, t >= 0, keep);
          cp_async16_hint(ddOb + off, A.dout + grow, t >= 0, keep);
        }
        sh->nlse2[sl][r0 + lane] = -mcur.x;
        sh->ndrow[sl][r0 + lane] = -mcur.y * d.scale;
        if (gw == 0) sh->tok[sl][lane] = tcur;
        cp_async_arrive(&sh->q_full[sl]);
        mbar_arrive(&sh->q_full[sl]);  // publishes the row data and tok
        tcur = tnext;
        mcur = mnext;
      }
    }
    cp_async_wait_all();  // nothing may land after the block exits
  } else if (warp == 3) {
    // ---------------------------------------------------------------- dQ reducer
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();  // dQ rows of the chunk: reduced into again
      long long ns = 0;
      for (long long ni = 0; ok; ++ni) {
        int it;
        if (!take_item1(ni, it)) { ok = false; break; }
        if (it >= total) break;
        const Item item = A.items[it];
        const int bg = (int)((item.seg % d.nseg()) / d.nblk);
        const int b = bg / d.Hp, a = (bg % d.Hp) * d.R + item.sub;
        const int ntiles = (item.count + TT - 1) / TT;
        for (int tl = 0; tl < ntiles; ++tl, ++ns) {
          const int sl = (int)(ns % kQSW);
          if (!wait1(11, &sh->stage_ready[sl], par(ns / kQSW))) { ok = false; break; }
          const uint32_t aSt = aSl + (uint32_t)sl * kSlotW;  // the tile's dQ rows, staged in its slot
#pragma unroll 1
          for (int x = 0; x < TT; ++x) {
            const int t = sh->tok[sl][x];
            if (t >= 0)
              bulk_reduce_add(A.dq + (((size_t)b * d.S + t) * d.Hq + a * G) * kD,
                              aSt + x * G * kD * 4, G * kD * 4, keep);
          }
          bulk_commit();
          bulk_wait_read0();
          mbar_arrive(&sh->q_empty[sl]);  // the slot may take the rows of tile ns + kQSW
        }
      }
      bulk_wait0();
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax / epilogue
    // Warps 4-7 take the tile's rows 0-63 (chunks 0, 1 of 32 rows) and the item's dV, warps 8-11
    // rows 64-127 (chunks 2, 3) and dK; warp w reads tensor-memory lanes 32 (w % 4) onwards.
    const int hf = (warp - 4) >> 2;  // half of the tile
    const int quad = warp & 3;
    const int kr = quad * 32 + lane;  // key row of S^T / dP^T (TMEM lane); head-dim index of dQ^T
    const uint32_t lb = static_cast<uint32_t>(quad * 32) << 16;
    const uint64_t stream = l2_policy_evict_first();  // pbar rows: read once, by proxy_bwd
    long long i = 0;
    for (long long ni = 0; ok; ++ni) {
      int it;
      if (!take_itemw(ni, it)) { ok = false; break; }
      if (it >= total) break;
      const Item item = A.items[it];
      const int n = item.seg % d.nblk;
      const int bg = (int)((item.seg % d.nseg()) / d.nblk);
      const int b = bg / d.Hp, kvh = d.kv_of((bg % d.Hp) * d.R + item.sub);
      const int j = n * kBlock + kr;  // this thread's key
      const long long eb = (long long)A.seg_offset[item.seg] + item.first;  // first list entry
      const int ntiles = (item.count + TT - 1) / TT;
      for (int tl = 0; tl < ntiles; ++tl, ++i) {
        const int sl = (int)(i % kQSW);
        __syncwarp();
        if (!waitw(12, &sh->q_full[sl], par(i / kQSW)) || !waitw(13, &sh->s_full, par(i))) {
          ok = false;
          break;
        }
        fence_after_sync();
        // ---- softmax of tile i: 32 rows at a time (P^T of rows 32 c .. 32 c + 31 lands in
        // columns 16 c + 32 hf .. + 15, which this half's first chunk has already read).  G divides
        // 32, so the G rows of a token lie in one chunk: each chunk finishes the teacher rows of
        // its tokens.
        constexpr int WT = 32 / G;  // tokens per chunk
#pragma unroll 1
        for (int c = 2 * hf; c < 2 * hf + 2; ++c) {
          float pc[WT];
          bool vis[WT];  // this thread's key is visible to the chunk's token w
#pragma unroll
          for (int w = 0; w < WT; ++w) {
            const int t = sh->tok[sl][c * WT + w];
            vis[w] = t >= 0 && j <= t;
            pc[w] = 0.f;
          }
          const uint32_t panel = adS + (uint32_t)(c >> 1) * (128 * 128);
          const float2 sl2x2 = make_float2(sl2, sl2), sc2 = make_float2(d.scale, d.scale);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {  // 16 rows at a time (fewer live registers)
            uint32_t rs[16], rp[16], pw[8], dw[8];
            __syncwarp();
            tmem_ld16(SB + lb + 32 * c + 16 * hh, rs);
            tmem_ld16(DB + lb + 32 * c + 16 * hh, rp);
            tmem_wait_ld();
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              const int q4 = hh * 4 + qq;
              const float4 l4 = reinterpret_cast<const float4*>(sh->nlse2[sl])[c * 8 + q4];
              const float4 d4 = reinterpret_cast<const float4*>(sh->ndrow[sl])[c * 8 + q4];
              const float nl[4] = {l4.x, l4.y, l4.z, l4.w};
              const float nd[4] = {d4.x, d4.y, d4.z, d4.w};
              float pv[4], dsv[4];
#pragma unroll
              for (int e = 0; e < 4; e += 2) {  // two rows per packed instruction
                const int r = qq * 4 + e;      // row within the 16
                const float2 x = ffma2(make_float2(__uint_as_float(rs[r]), __uint_as_float(rs[r + 1])),
                                       sl2x2, make_float2(nl[e], nl[e + 1]));
                pv[e] = vis[(q4 * 4 + e) / G] ? ex2(x.x) : 0.f;
                pv[e + 1] = vis[(q4 * 4 + e + 1) / G] ? ex2(x.y) : 0.f;
                // dS = scale P (dP - D): the softmax scale of dK and dQ is folded in here
                const float2 ds = fmul2(make_float2(pv[e], pv[e + 1]),
                                        ffma2(make_float2(__uint_as_float(rp[r]), __uint_as_float(rp[r + 1])),
                                              sc2, make_float2(nd[e], nd[e + 1])));
                dsv[e] = ds.x;
                dsv[e + 1] = ds.y;
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) pc[(q4 * 4 + e) / G] += pv[e];  // the token's G heads
              pw[2 * qq] = pack_bf16(pv[0], pv[1]);
              pw[2 * qq + 1] = pack_bf16(pv[2], pv[3]);
              dw[2 * qq] = pack_bf16(dsv[0], dsv[1]);
              dw[2 * qq + 1] = pack_bf16(dsv[2], dsv[3]);
            }
            // P^T and dS^T of these 16 rows: 8 columns of bf16 pairs each, over columns of S^T
            // and dP^T this half has read (dS^T also goes to shared memory for dQ^T below)
            tmem_st8(SB + lb + 16 * c + 32 * hf + 8 * hh, pw);
            tmem_st8(DB + lb + 16 * c + 32 * hf + 8 * hh, dw);
#pragma unroll
            for (int u = 0; u < 2; ++u)
              st_shared_v4(panel + sm100::sw128_chunk(kr, (c & 1) * 4 + 2 * hh + u), dw[4 * u],
                           dw[4 * u + 1], dw[4 * u + 2], dw[4 * u + 3]);
          }
          // teacher: mean of the proxy head's G R query heads' probabilities of each token, one
          // fp16 row per list entry; with R > 1 attention groups per proxy head each adds its share
          if (d.R == 1) {
#pragma unroll
            for (int w = 0; w < WT; ++w)
              if (sh->tok[sl][c * WT + w] >= 0)
                st_global_h_hint(A.pbar + (size_t)(eb - ent0 + tl * TT + c * WT + w) * kBlock + kr,
                                 pc[w] * (1.f / G), stream);
          } else {
#pragma unroll
            for (int w = 0; w < WT; ++w)
              if (sh->tok[sl][c * WT + w] >= 0)
                red_add_h(A.pbar + (size_t)(eb - ent0 + tl * TT + c * WT + w) * kBlock + kr,
                          pc[w] * (1.f / (G * d.R)));
          }
        }
        __syncwarp();
        tmem_wait_st();
        fence_async_smem();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->p_full);
        // ---- epilogue of tile i: dQ^T -> fp32 rows staged in the tile's own slot (phase 2 has
        // finished reading its Q / dO rows); the reducer then adds them to dQ
        __syncwarp();
        if (!waitw(14, &sh->ph2_full, par(i))) { ok = false; break; }
        fence_after_sync();
        float* stage = reinterpret_cast<float*>(sSl + sl * kSlotW);
        {
          // both chunks of this half out of DB first, so that DB is free for the next tile's dP^T
          // before the rows are staged
          uint32_t r0[32], r1[32];
          __syncwarp();
          tmem_ld32(DB + lb + 64 * hf, r0);
          tmem_ld32(DB + lb + 64 * hf + 32, r1);
          tmem_wait_ld();
          fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh->s_free);
#pragma unroll
          for (int r = 0; r < 32; ++r) stage[(64 * hf + r) * kD + kr] = __uint_as_float(r0[r]);
#pragma unroll
          for (int r = 0; r < 32; ++r) stage[(64 * hf + 32 + r) * kD + kr] = __uint_as_float(r1[r]);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->stage_ready[sl]);
      }
      if (!ok) break;
      // ---- item end: dV (rows-0-63 warps) or dK (rows-64-127 warps) row of this key (the
      // item's last phase 2 has completed)
      {
        float* dst = (hf == 0 ? A.dv : A.dk) + (((size_t)b * d.S + j) * d.Hkv + kvh) * kD;
        const uint32_t acc_t = hf == 0 ? RV : RK;
        __syncwarp();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t rv[32];
          tmem_ld32(acc_t + lb + c * 32, rv);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 8; ++u)
            red4(dst + c * 32 + 4 * u, __uint_as_float(rv[4 * u]), __uint_as_float(rv[4 * u + 1]),
                 __uint_as_float(rv[4 * u + 2]), __uint_as_float(rv[4 * u + 3]));
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->acc_free);
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) {
    waitw(15, &sh->mma_done, 0);  // no MMA may still write tensor memory when it is freed
    tmem_dealloc(tmem, 512);
  }
}

// ==========================================================================================
// Proxy gradients of the KL term from the teacher pbar written by attn_bwd_kernel.
// Roles (384 threads): warp 0 TMA of the block's proxy keys + tensor memory, warp 1 MMA, warps 2-3
// gather the group's Qp rows and pbar rows, warps 4-7 compute dz (thread = key) and flush dKp at
// item end, warps 8-11 flush dQp.  Tensor memory (512 columns allocated): Z0, Z1 (z^T, 64 each,
// alternate groups), QP (dQp^T, 64), KP (dKp accumulator, 128).  dz^T is double-buffered in
// shared memory, so the dz of one group overlaps the products and the flush of the previous one.
template <bool kDense, bool kKL>
__global__ void __launch_bounds__(384, 1)
    proxy_bwd_kernel(const __grid_constant__ CUtensorMap tm_kp, const __grid_constant__ CUtensorMap tm_qp,
                     const __grid_constant__ CUtensorMap tm_dqp, ProxyArgs A) {
  using namespace sm100;
  const Dims& d = A.d;
  extern __shared__ uint8_t smem_raw[];
  ProxyShared* sh = reinterpret_cast<ProxyShared*>(smem_raw);
  uint8_t* base = align1024(smem_raw + sizeof(ProxyShared));
  uint8_t* sKp = base;             // [128 keys][128 d]  (TMA)
  uint8_t* sQp = sKp + kKV;        // [kQPB][64 tokens][128 d]
  uint8_t* sdz = sQp + kQPB * kRT;  // [2] dz^T [128 keys][64 tokens]
  __half* sPb = reinterpret_cast<__half*>(sdz + 2 * kST);  // [kNPB][64 entries][128 keys] fp16
  float* sStg = reinterpret_cast<float*>(sPb + kNPB * kPG * kBlock);  // dQp staging: [4 warps][64 tokens][32 d]
  const uint32_t aKp = smem_u32(sKp), aQp = smem_u32(sQp), adz = smem_u32(sdz);

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const float sl2 = d.scale * kLog2e;
  const float cz = A.czp ? A.cz * __ldg(A.czp) : A.cz;
  long long total = A.item_hi ? *A.item_hi : *A.n_items;  // items of this pass end here
  if (total > A.max_items) total = A.max_items;
  const int item0 = A.item_lo ? *A.item_lo : 0;
  const long long ent0 = A.entry_lo ? *A.entry_lo : 0;  // list entry of teacher row 0
  if (tid == 0) {
    mbar_init(&sh->kp_full, 1);
    mbar_init(&sh->kp_empty, 1);
    for (int x = 0; x < kQPB; ++x) {
      mbar_init(&sh->qp_full[x], 128);  // 2 gather warps x 32 lanes: a plain and a cp.async arrival
      mbar_init(&sh->qp_empty[x], 5);   // the MMA's commit and the 4 dQp-flush warps
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sh->z_full[x], 1);
      mbar_init(&sh->fl_full[x], 1);
    }
    for (int x = 0; x < kNPB; ++x) {
      mbar_init(&sh->pb_full[x], 64);   // the gather lanes (one with the bulk copy's expect-tx)
      mbar_init(&sh->meta_free[x], 4);  // the dz warps
    }
    mbar_init(&sh->dz_full, 4);
    mbar_init(&sh->fl_free, 4);
    mbar_init(&sh->acc_free, 4);
    for (int x = 0; x < kIR; ++x) {
      mbar_init(&sh->it_full[x], 1);
      mbar_init(&sh->it_empty[x], 11);  // MMA, 2 gather warps, 4 dz warps, 4 flush warps
    }
    mbar_fence_init();
  }
  if (warp == 0) {
    __syncwarp();  // lane 0 initialised the barriers alone; the allocation is warp-collective
    tmem_alloc(&sh->tmem, 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sh->tmem;
  const uint32_t RZ0 = tmem, RQ = tmem + 128, RKP = tmem + 256;  // RZ_b = RZ0 + 64 b
  bool ok = true;
  // item number ni of this block (handed out in list order by a shared counter), for one thread /
  // for a whole warp
  auto take_item1 = [&](long long ni, int& v) -> bool {
    const int x = (int)(ni % kIR);
    if (!mbar_wait(&sh->it_full[x], par(ni / kIR), A.status)) return false;
    v = sh->it_ring[x];
    mbar_arrive(&sh->it_empty[x]);
    return true;
  };
  auto take_itemw = [&](long long ni, int& v) -> bool {
    const int x = (int)(ni % kIR);
    if (!mbar_wait_warp(&sh->it_full[x], par(ni / kIR), A.status)) return false;
    v = sh->it_ring[x];
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh->it_empty[x]);
    return true;
  };

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_kp);
      // item numbers are published up to two items ahead of the proxy-key loads
      long long pub = 0;
      bool last = false;
      for (long long ni = 0;; ++ni) {
        while (!last && pub < ni + 2) {
          const int x = (int)(pub % kIR);
          if (pub >= kIR && !mbar_wait(&sh->it_empty[x], par(pub / kIR - 1), A.status)) break;
          // the work items repeat each run of tokens for the proxy head's R attention groups;
          // the proxy gradients need each run once
          int v = item0 + atomicAdd(A.sched, 1);
          while (v < total && A.items[v].sub != 0) v = item0 + atomicAdd(A.sched, 1);
          sh->it_ring[x] = v;
          mbar_arrive(&sh->it_full[x]);
          last = v >= total;
          ++pub;
        }
        if (pub <= ni) break;  // a wait gave up
        const int it = sh->it_ring[ni % kIR];
        if (it >= total) break;
        const Item item = A.items[it];
        const int n = item.seg % d.nblk;
        const int bg = (int)((item.seg % d.nseg()) / d.nblk);
        const int b = bg / d.Hp;
        if (ni > 0 && !mbar_wait(&sh->kp_empty, par(ni - 1), A.status)) break;
        mbar_expect_tx(&sh->kp_full, kKV);
        tma_load_2d(sKp, &tm_kp, 0, b * d.S + n * kBlock, &sh->kp_full);
        tma_load_2d(sKp + kKV / 2, &tm_kp, 64, b * d.S + n * kBlock, &sh->kp_full);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: z(i) for group i, then the gradients of group i-1 (within an item)
    if (lane == 0) {
      constexpr uint32_t id_z = idesc_bf16(128, kPG, false, false);
      constexpr uint32_t id_k = idesc_bf16(128, 128, false, true);
      constexpr uint32_t id_p = idesc_bf16(128, kPG, true, true);
      long long ni = 0, i = 0;
      // dKp += dz^T Qp and dQp^T = Kp^T dz^T for group j (gj-th of its item, gcount tokens)
      auto grads = [&](long long j, int gj, int gcount, bool last) -> bool {
        const int b = (int)(j & 1);
        if (!mbar_wait(&sh->dz_full, par(j), A.status)) return false;
        if (gj == 0 && ni > 0 && !mbar_wait(&sh->acc_free, par(ni - 1), A.status)) return false;
        if (j > 0 && !mbar_wait(&sh->fl_free, par(j - 1), A.status)) return false;  // RQ read
        fence_async_smem();  // dz^T was written with st.shared by the dz warps
        fence_after_sync();
        const uint32_t aQb = aQp + (int)(j % kQPB) * kRT, adzb = adz + b * kST;
        const int kst = (gcount + 15) / 16;
        for (int ks = 0; ks < kst; ++ks)  // dKp += dz^T Qp
          mma_ss(RKP, desc_kmajor(adzb, 128, ks), desc_mnmajor(aQb, kPG, ks), id_k, gj > 0 || ks > 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)  // dQp^T = Kp^T dz^T
          mma_ss(RQ, desc_mnmajor(aKp, 128, ks), desc_mnmajor(adzb, 128, ks), id_p, ks > 0);
        mma_commit(&sh->fl_full[b]);
        mma_commit(&sh->qp_empty[j % kQPB]);
        if (last) mma_commit(&sh->kp_empty);
        return true;
      };
      for (;; ++ni) {
        int it;
        if (!take_item1(ni, it)) { ok = false; break; }
        if (it >= total) break;
        const Item item = A.items[it];
        if (!mbar_wait(&sh->kp_full, par(ni), A.status)) { ok = false; break; }
        const int ngroups = (item.count + kPG - 1) / kPG;
        for (int gi = 0; gi < ngroups; ++gi, ++i) {
          const int b = (int)(i & 1), qb = (int)(i % kQPB);
          if (!mbar_wait(&sh->qp_full[qb], par(i / kQPB), A.status)) { ok = false; break; }
          // RZ_b was last read by the dz warps for group i-2; the gradients of that group, which
          // waited for it (dz_full), were issued before this point
          // Qp rows came from other threads' cp.async (generic proxy), tracked by qp_full
          fence_async_smem();
          fence_after_sync();
          const uint32_t aQb = aQp + qb * kRT;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // z^T = Kp Qp^T
            mma_ss(RZ0 + 64 * b, desc_kmajor(aKp, 128, ks), desc_kmajor(aQb, kPG, ks), id_z, ks > 0);
          mma_commit(&sh->z_full[b]);
          if (gi > 0 && !grads(i - 1, gi - 1, kPG, false)) { ok = false; break; }
        }
        if (!ok) break;
        if (ngroups > 0 &&
            !grads(i - 1, ngroups - 1, item.count - (ngroups - 1) * kPG, true)) { ok = false; break; }
      }
    }
  } else if (warp == 2 || warp == 3) {
    // ---- gather: warp 2 + w handles rows 32 w .. 32 w + 31 of each group.  The group's teacher
    // rows (consecutive list entries, so contiguous) come with one bulk copy issued by lane 0 of
    // warp 2 as soon as the dz warps have released that buffer; the proxy query rows come with
    // cp.async into one of three buffers, released by the MMA and the dQp-flush warps.  The next
    // group's tokens and proxy normalisers are loaded one step ahead.
    const int w = warp - 2;
    long long gni = 0;
    int it = 0;
    if (!take_itemw(gni, it)) ok = false;
    if (ok && it < total) {
      Item cur = A.items[it];
      int gi = 0;
      // token and proxy log-normaliser (x log2 e) of group row 32 w + lane of group `grp`
      auto load_row = [=](const Item& item, int grp, float& lp) -> int {
        const int bg = (int)((item.seg % d.nseg()) / d.nblk);
        const int b = bg / d.Hp, g = bg % d.Hp;
        const int x = 32 * w + lane;
        const int pos = grp * kPG + x;
        int t = -1;
        lp = 0.f;
        if (pos < item.count) {
          if (kDense) {  // consecutive tokens: the row's normaliser by token
            t = (int)(item_base<true>(d, nullptr, item) + pos);
            lp = __ldg(A.lse_px + (size_t)bg * d.S + t) * kLog2e;
          } else {  // two independent loads, both indexed by the entry
            t = __ldg(A.entries + item.base + pos) >> 8;
            lp = __ldg(A.lpxe + item.base + pos);
          }
        }
        (void)b;
        (void)g;
        return t;
      };
      float lp_next;
      int t_next = load_row(cur, 0, lp_next);
      long long i = 0;
      while (true) {
        const int pb = (int)(i % kNPB), qb = (int)(i % kQPB);
        const int gcount = min(kPG, cur.count - gi * kPG);
        // ---- teacher rows + dz metadata (buffer pb: free once the dz warps read group i-kNPB)
        if (i >= kNPB && !mbar_wait_warp(&sh->meta_free[pb], par(i / kNPB - 1), A.status)) {
          ok = false;
          break;
        }
        sh->tok[pb][32 * w + lane] = t_next;
        sh->lpx2[pb][32 * w + lane] = lp_next;
        __syncwarp();
        if (w == 0 && lane == 0) {  // gcount entries x 128 keys, one bulk copy
          const uint32_t bytes = (uint32_t)gcount * kBlock * 2;
          mbar_expect_tx(&sh->pb_full[pb], bytes);  // also this lane's arrival
          bulk_load(sPb + pb * kPG * kBlock, A.pbar + (size_t)(cur.base - ent0 + gi * kPG) * kBlock, bytes,
                    &sh->pb_full[pb]);
        } else {
          mbar_arrive(&sh->pb_full[pb]);  // publishes tok / lpx2
        }
        // ---- proxy query rows (buffer qb: free once group i-3's products and flush are done)
        if (i >= kQPB && !mbar_wait_warp(&sh->qp_empty[qb], par(i / kQPB - 1), A.status)) {
          ok = false;
          break;
        }
        const int bg = (int)((cur.seg % d.nseg()) / d.nblk);
        const int b = bg / d.Hp, g = bg % d.Hp;
        sh->tokq[qb][32 * w + lane] = t_next;
        __syncwarp();
        uint8_t* dQb = sQp + qb * kRT;
        if constexpr (kDense) {
          // a dense group's tokens are consecutive (t_next of row 0 is the first): its proxy query
          // rows come with two TMA boxes of 64 rows, one per 64-column panel (rows beyond the
          // group's tokens load other rows -- their dz is zero -- or the fill value past the end)
          if (w == 0 && lane == 0) {
            mbar_expect_tx(&sh->qp_full[qb], kPG * kD * 2);  // also this lane's first arrival
            tma_load_3d(dQb, &tm_qp, 0, g, b * d.S + t_next, &sh->qp_full[qb]);
            tma_load_3d(dQb + kPG * 128, &tm_qp, 64, g, b * d.S + t_next, &sh->qp_full[qb]);
          } else {
            mbar_arrive(&sh->qp_full[qb]);
          }
          mbar_arrive(&sh->qp_full[qb]);  // publishes tokq
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) {  // K-major SW128 rows, rows >= gcount zero-filled
            const int c = lane + 32 * k;  // 16-byte chunk of this warp's 32 rows
            const int r = 32 * w + (c >> 4), ch = c & 15;
            const int t = sh->tokq[qb][r];
            const uint32_t off = (ch >> 3) * (kPG * 128) + sm100::sw128_chunk(r, ch & 7);
            const size_t grow = (((size_t)b * d.S + (t < 0 ? 0 : t)) * d.Hp + g) * kD + ch * 8;
            cp_async16(dQb + off, A.qp + grow, t >= 0);
          }
          cp_async_arrive(&sh->qp_full[qb]);
          mbar_arrive(&sh->qp_full[qb]);  // publishes tokq
        }
        ++i;
        const int ngroups = (cur.count + kPG - 1) / kPG;
        if (gi + 1 < ngroups) {
          ++gi;
          t_next = load_row(cur, gi, lp_next);
        } else {
          if (!take_itemw(++gni, it)) { ok = false; break; }
          if (it >= total) break;
          cur = A.items[it];
          gi = 0;
          t_next = load_row(cur, 0, lp_next);
        }
      }
      cp_async_wait_all();  // nothing may land after the block exits
      // the last bulk copies land before the block exits
      for (long long x = (i >= kNPB ? i - kNPB : 0); x < i; ++x)
        mbar_wait_warp(&sh->pb_full[x % kNPB], par(x / kNPB), A.status);
    }
  } else if (warp < 8) {
    // ---- dz (thread = key): dz^T = kl_grad/(B S Hp) (softmax(scale z) - pbar); item end: dKp
    const int w4 = warp - 4;
    const int kr = w4 * 32 + lane;  // key (tensor-memory lane of z^T and dKp)
    const uint32_t lb = static_cast<uint32_t>(w4 * 32) << 16;
    float kl = 0.f;  // kKL: this thread's share of sum pbar (ln pbar - ln p_student)
    long long i = 0;
    for (long long ni = 0; ok; ++ni) {
      int it;
      if (!take_itemw(ni, it)) { ok = false; break; }
      if (it >= total) break;
      const Item item = A.items[it];
      const int n = item.seg % d.nblk;
      const int bg = (int)((item.seg % d.nseg()) / d.nblk);
      const int b = bg / d.Hp;
      const int j = n * kBlock + kr;
      const int ngroups = (item.count + kPG - 1) / kPG;
      for (int gi = 0; gi < ngroups; ++gi, ++i) {
        const int bb = (int)(i & 1), pbi = (int)(i % kNPB);
        const int gcount = min(kPG, item.count - gi * kPG);
        __syncwarp();
        if (!mbar_wait_warp(&sh->pb_full[pbi], par(i / kNPB), A.status) ||
            !mbar_wait_warp(&sh->z_full[bb], par(i >> 1), A.status)) {
          ok = false;
          break;
        }
        // dz^T buffer bb was last read by the gradient products of group i-2, which ran on the
        // tensor core before z of this group (already complete: z_full)
        if (i >= 2 && !mbar_wait_warp(&sh->fl_full[bb], par((i - 2) >> 1), A.status)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const __half* pbr = sPb + pbi * kPG * kBlock;
        const uint32_t adzb = adz + bb * kST;
        const float2 sl2x2 = make_float2(sl2, sl2), cz2 = make_float2(cz, cz);
#pragma unroll 1
        for (int h16 = 0; h16 < kPG / 16; ++h16) {  // 16 tokens (two 16-byte chunks of dz^T) at a time
          uint32_t zr[16], zw[8];
          __syncwarp();
          tmem_ld16(RZ0 + 64 * bb + lb + 16 * h16, zr);
          tmem_wait_ld();
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int kb = 16 * h16 + 4 * k4;
            const int4 t4 = *reinterpret_cast<const int4*>(&sh->tok[pbi][kb]);
            const float4 l4 = *reinterpret_cast<const float4*>(&sh->lpx2[pbi][kb]);
            const int tv[4] = {t4.x, t4.y, t4.z, t4.w};
            const float nl[4] = {-l4.x, -l4.y, -l4.z, -l4.w};
#pragma unroll
            for (int pp = 0; pp < 2; ++pp) {
              const int k = kb + 2 * pp;
              // log2 of the student probabilities; exponentiate unconditionally and select
              const float2 lz = ffma2(make_float2(__uint_as_float(zr[4 * k4 + 2 * pp]),
                                                  __uint_as_float(zr[4 * k4 + 2 * pp + 1])),
                                      sl2x2, make_float2(nl[2 * pp], nl[2 * pp + 1]));
              const float pb0 = __half2float(pbr[k * kBlock + kr]);
              const float pb1 = __half2float(pbr[(k + 1) * kBlock + kr]);
              const float2 v = fmul2(cz2, fadd2(make_float2(ex2(lz.x), ex2(lz.y)), make_float2(-pb0, -pb1)));
              const bool vis0 = k < gcount && tv[2 * pp] >= 0 && j <= tv[2 * pp];
              const bool vis1 = k + 1 < gcount && tv[2 * pp + 1] >= 0 && j <= tv[2 * pp + 1];
              zw[2 * k4 + pp] = pack_bf16(vis0 ? v.x : 0.f, vis1 ? v.y : 0.f);
              if constexpr (kKL) {
                kl += (vis0 && pb0 > 0.f) ? pb0 * (__logf(pb0) - lz.x * kLn2) : 0.f;
                kl += (vis1 && pb1 > 0.f) ? pb1 * (__logf(pb1) - lz.y * kLn2) : 0.f;
              }
            }
          }
          st_shared_v4(adzb + sm100::sw128_chunk(kr, 2 * h16), zw[0], zw[1], zw[2], zw[3]);
          st_shared_v4(adzb + sm100::sw128_chunk(kr, 2 * h16 + 1), zw[4], zw[5], zw[6], zw[7]);
        }
        fence_async_smem();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sh->dz_full);        // also: RZ_bb read
          mbar_arrive(&sh->meta_free[pbi]);  // tok / lpx2 / pbar rows of this buffer read
        }
        if (gi == ngroups - 1) {  // item end: dKp rows of this key, once its last product landed
          if (!mbar_wait_warp(&sh->fl_full[bb], par(i >> 1), A.status)) {
            ok = false;
            break;
          }
          fence_after_sync();
          float* dst = A.dkp + ((size_t)b * d.S + j) * kD;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            __syncwarp();
            uint32_t rk[32];
            tmem_ld32(RKP + lb + c * 32, rk);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 8; ++u)
              red4(dst + c * 32 + 4 * u, __uint_as_float(rk[4 * u]) * d.scale,
                   __uint_as_float(rk[4 * u + 1]) * d.scale, __uint_as_float(rk[4 * u + 2]) * d.scale,
                   __uint_as_float(rk[4 * u + 3]) * d.scale);
          }
          fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh->acc_free);
        }
      }
    }
    if constexpr (kKL) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) kl += __shfl_xor_sync(0xffffffffu, kl, off);
      if (lane == 0) atomicAdd(A.kl_acc, (double)kl);
    }
  } else {
    // ---- dQp flush (warps 8-11, thread = head-dim index): dQp^T -> token-major staging ->
    // 16-byte reductions, each instruction covering 4 tokens x 128 contiguous bytes
    const int w4 = warp - 8;
    const uint32_t lb = static_cast<uint32_t>(w4 * 32) << 16;
    float* stg = sStg + w4 * (kPG * 32);
    long long i = 0;
    for (long long ni = 0; ok; ++ni) {
      int it;
      if (!take_itemw(ni, it)) { ok = false; break; }
      if (it >= total) break;
      const Item item = A.items[it];
      const int bg = (int)((item.seg % d.nseg()) / d.nblk);
      const int b = bg / d.Hp, g = bg % d.Hp;
      const int ngroups = (item.count + kPG - 1) / kPG;
      for (int gi = 0; gi < ngroups; ++gi, ++i) {
        const int bb = (int)(i & 1), qb = (int)(i % kQPB);
        const int gcount = min(kPG, item.count - gi * kPG);
        __syncwarp();
        // (qp_full: acquire the gather's token list of this buffer; already complete)
        if (!mbar_wait_warp(&sh->fl_full[bb], par(i >> 1), A.status) ||
            !mbar_wait_warp(&sh->qp_full[qb], par(i / kQPB), A.status)) {
          ok = false;
          break;
        }
        fence_after_sync();
        uint32_t q0[32], q1[32];
        tmem_ld32(RQ + lb, q0);
        tmem_ld32(RQ + lb + 32, q1);
        tmem_wait_ld();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->fl_free);  // RQ may take the next group's dQp^T
#pragma unroll
        for (int k = 0; k < kPG; ++k)
          stg[k * 32 + lane] = __uint_as_float(k < 32 ? q0[k] : q1[k - 32]) * d.scale;
        __syncwarp();
        if constexpr (kDense) {
          // consecutive tokens: one TMA tensor reduction adds this warp's 64 tokens x 32 columns
          // (the rows beyond the group's tokens hold exact zeros: their dz is zero)
          fence_async_smem();  // the staging rows (generic-proxy stores) before the TMA reads them
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_3d(&tm_dqp, 32 * w4, g, b * d.S + sh->tokq[qb][0], smem_u32(stg));
            bulk_commit();
            bulk_wait_read0();  // the staging rows may be overwritten by the next group
          }
          __syncwarp();
        } else {
#pragma unroll 4
          for (int it2 = 0; it2 < kPG / 4; ++it2) {
            const int k = it2 * 4 + lane / 8, c4 = lane % 8;
            const float4 v = *reinterpret_cast<const float4*>(stg + k * 32 + 4 * c4);
            const int t = k < gcount ? sh->tokq[qb][k] : -1;
            red_add_v4_if(t >= 0,
                          A.dqp + (((size_t)b * d.S + (t < 0 ? 0 : t)) * d.Hp + g) * kD + w4 * 32 + 4 * c4, v);
          }
          __syncwarp();
        }
        if (lane == 0) mbar_arrive(&sh->qp_empty[qb]);  // token list of this buffer read
      }
    }
    if constexpr (kDense) {
      if (lane == 0) bulk_wait0();  // every reduction has landed before the block exits
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

namespace {
template <int G, bool kDense>
void attn_bwd_g(const CUtensorMap& mk, const CUtensorMap& mv, const MainArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(MainShared) + 1024 + 2 * (size_t)kKV + kQS * (size_t)kSlot +
                      2 * (size_t)kST;
  cudaFuncSetAttribute(attn_bwd_kernel<G, kDense>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smem);
  attn_bwd_kernel<G, kDense><<<num_sms(), 352, smem, st>>>(mk, mv, a);
}
template <int G, bool kDense>
void attn_bwd_wide_g(const CUtensorMap& mk, const CUtensorMap& mv, const MainArgs& a, cudaStream_t st) {
  const size_t smem = kWideSmem + sizeof(WideShared);  // base 1024-aligned (checked in the kernel)
  cudaFuncSetAttribute(attn_bwd_wide_kernel<G, kDense>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smem);
  attn_bwd_wide_kernel<G, kDense><<<num_sms(), kWideThreads, smem, st>>>(mk, mv, a);
}
template <bool kDense, bool kKL>
void proxy_bwd_g(const CUtensorMap& mkp, const CUtensorMap& mqp, const CUtensorMap& mdqp,
                 const ProxyArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(ProxyShared) + 1024 + (size_t)kKV + kQPB * (size_t)kRT + 2 * (size_t)kST +
                      kNPB * (size_t)kPG * kBlock * 2 + 4 * (size_t)kPG * 32 * 4;
  cudaFuncSetAttribute(proxy_bwd_kernel<kDense, kKL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smem);
  proxy_bwd_kernel<kDense, kKL><<<num_sms(), 384, smem, st>>>(mkp, mqp, mdqp, a);
}

__global__ void kl_finalize_kernel(const double* acc, float* out, double inv) {
  out[0] = (float)(acc[0] * inv);
}
}  // namespace

int bwd_item_tokens() { return kItemTokens; }
int bwd_group_tokens() { return kPG; }

void launch_bwd_rowdot(const Dims& d, const void* o, const void* dout, const float* lse,
                       float2* rowm, cudaStream_t st) {
  const long long rows = (long long)d.B * d.S * d.Hq;
  long long grid = ((rows + 3) / 4 * 32 + 255) / 256;
  if (grid > (long long)num_sms() * 16) grid = (long long)num_sms() * 16;
  rowdot_kernel<<<(int)grid, 256, 0, st>>>(d, (const bf16*)o, (const bf16*)dout, lse, rowm);
}

bool launch_attn_bwd(const Dims& d, bool dense, const void* q, const void* k, const void* v,
                     const void* dout, const float2* rowdata, const int* seg_offset,
                     const int* entries, const Item* items, const int* n_items, long long max_items,
                     const int* item_lo, const int* item_hi, const int* entry_lo,
                     float* dq_acc, float* dk_acc, float* dv_acc, void* pbar, unsigned* status,
                     cudaStream_t st) {
  CUtensorMap mk, mv;
  const uint64_t kvd[3] = {128, (uint64_t)d.Hkv, (uint64_t)d.B * d.S};
  const uint64_t kvs[2] = {128 * 2, (uint64_t)d.Hkv * 128 * 2};
  const uint32_t kvb[3] = {64, 1, 128};
  if (!make_tmap_bf16(&mk, k, 3, kvd, kvs, kvb) || !make_tmap_bf16(&mv, v, 3, kvd, kvs, kvb))
    return false;
  MainArgs a;
  a.d = d;
  a.q = (const bf16*)q;
  a.dout = (const bf16*)dout;
  a.emeta = dense ? nullptr : rowdata;
  a.rowm = dense ? rowdata : nullptr;
  a.seg_offset = seg_offset;
  a.entries = entries;
  a.items = items;
  a.n_items = n_items;
  a.max_items = max_items;
  a.dq = dq_acc;
  a.dk = dk_acc;
  a.dv = dv_acc;
  a.pbar = static_cast<__half*>(pbar);
  a.status = status;
  a.sched = reinterpret_cast<int*>(status + kSchedAttnBwd);
  a.item_lo = item_lo;
  a.item_hi = item_hi;
  a.entry_lo = entry_lo;
  cudaMemsetAsync(a.sched, 0, sizeof(int), st);
  // 128-row tiles for 4 and 8 heads per group; 16 heads keep 64-row tiles (there P and dS go to
  // the products as a bf16 value plus its bf16 residual, which needs the spare tensor memory).
  // The dense mode with 8 heads per group also keeps the 64-row kernel: its 128-row instance
  // raised an illegal-instruction fault on a 512-token case whose cause is not yet found.
  switch (d.G) {
    case 4:
      dense ? attn_bwd_wide_g<4, true>(mk, mv, a, st) : attn_bwd_wide_g<4, false>(mk, mv, a, st);
      break;
    case 8:
      dense ? attn_bwd_g<8, true>(mk, mv, a, st) : attn_bwd_wide_g<8, false>(mk, mv, a, st);
      break;
    case 16:
      dense ? attn_bwd_g<16, true>(mk, mv, a, st) : attn_bwd_g<16, false>(mk, mv, a, st);
      break;
    default:
      return false;
  }
  return true;
}

bool launch_proxy_bwd(const Dims& d, bool dense, const void* qp, const void* kp,
                      const float* lpx, const void* pbar, float kl_grad,
                      const float* kl_grad_dev, const int* seg_offset,
                      const int* entries, const Item* items, const int* n_items,
                      long long max_items, const int* item_lo, const int* item_hi,
                      const int* entry_lo, float* dqp_acc, float* dkp_acc, double* kl_acc,
                      unsigned* status, cudaStream_t st) {
  CUtensorMap mkp;
  const uint64_t kpd[2] = {128, (uint64_t)d.B * d.S};
  const uint64_t kps[1] = {128 * 2};
  const uint32_t kpb[2] = {64, 128};
  if (!make_tmap_bf16(&mkp, kp, 2, kpd, kps, kpb)) return false;
  // dense groups (consecutive tokens): their proxy query rows and dQp rows as [B S][Hp][128]
  CUtensorMap mqp = mkp, mdqp = mkp;  // (unused by the sparse kernel)
  if (dense) {
    const uint64_t qd[3] = {128, (uint64_t)d.Hp, (uint64_t)d.B * d.S};
    const uint64_t qs[2] = {128 * 2, (uint64_t)d.Hp * 128 * 2};
    const uint32_t qb[3] = {64, 1, (uint32_t)kPG};
    const uint64_t fs[2] = {128 * 4, (uint64_t)d.Hp * 128 * 4};
    const uint32_t fb[3] = {32, 1, (uint32_t)kPG};
    if (!make_tmap_bf16(&mqp, qp, 3, qd, qs, qb) || !make_tmap_f32(&mdqp, dqp_acc, qd, fs, fb))
      return false;
  }
  ProxyArgs a;
  a.d = d;
  a.qp = (const bf16*)qp;
  a.lpxe = dense ? nullptr : lpx;
  a.lse_px = dense ? lpx : nullptr;
  a.pbar = static_cast<const __half*>(pbar);
  const double inv_n = 1.0 / ((double)d.B * d.S * d.Hp);
  a.cz = (float)(kl_grad_dev ? inv_n : (double)kl_grad * inv_n);
  a.czp = kl_grad_dev;
  a.seg_offset = seg_offset;
  a.entries = entries;
  a.items = items;
  a.n_items = n_items;
  a.max_items = max_items;
  a.dqp = dqp_acc;
  a.dkp = dkp_acc;
  a.kl_acc = kl_acc;
  a.status = status;
  a.sched = reinterpret_cast<int*>(status + kSchedProxyBwd);
  a.item_lo = item_lo;
  a.item_hi = item_hi;
  a.entry_lo = entry_lo;
  cudaMemsetAsync(a.sched, 0, sizeof(int), st);
  if (dense)
    kl_acc ? proxy_bwd_g<true, true>(mkp, mqp, mdqp, a, st) : proxy_bwd_g<true, false>(mkp, mqp, mdqp, a, st);
  else
    kl_acc ? proxy_bwd_g<false, true>(mkp, mqp, mdqp, a, st) : proxy_bwd_g<false, false>(mkp, mqp, mdqp, a, st);
  return true;
}

void launch_kl_finalize(const Dims& d, const double* kl_acc, float* kl_out, cudaStream_t st) {
  kl_finalize_kernel<<<1, 1, 0, st>>>(kl_acc, kl_out, 1.0 / ((double)d.B * d.S * d.Hp));
}

}  // namespace msa
