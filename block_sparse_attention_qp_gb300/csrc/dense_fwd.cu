// Dense causal forward of the warmup mode on the tcgen05 tensor cores (blog, "Warmup kernels":
// in warmup the main attention forward is dense over the causal prefix and the proxy forward is
// skipped).
//
// Q-outer: a work unit is one (b, group g, query block m) and a pair of 128-row query tiles of that
// block (a tile is 128/G consecutive tokens x the G query heads of the group, loaded by TMA); both
// tiles attend to key blocks 0 .. m (block m with the causal cut j <= t), so they share every K / V
// block of a four-slot TMA ring.  Per key block n and tile X in {A, B}:
//   S_X  = Q_X K_n^T                      (tensor core -> tensor memory, 128 x 128 fp32)
//   softmax warps (thread = row): running maximum mr of the raw scores; P = 2^(sl2 (S - mr)) in
//        bf16 over S in tensor memory, l += row sum.  mr only moves when the block maximum exceeds
//        it by more than 8 / sl2 (P stays <= 2^8); then O_X and l are first rescaled by
//        2^(sl2 (mr_old - mr_new)).  O_X's previous product has finished by then: it was issued
//        before S_X, and S_X's completion covers every earlier product.
//   O_X += P V_n                          (P read from tensor memory)
// Unit end: O_X / l -> bf16 rows, LSE = ln 2 (sl2 mr + log2 l).
// MMA issue order: S_A(0) S_B(0) | O_A(0) S_A(1) | O_B(0) S_B(1) | O_A(1) S_A(2) | ..., so the
// softmax of one tile runs while the tensor core works on the other.
// Roles (384 threads): warp 0 takes the work units (a shared counter, longest units first) and
// issues the TMA loads, warp 1 issues the MMAs (lane 0), warps 4-7 / 8-11 are the softmax and
// epilogue of tile A / B (warp w reads tensor-memory lanes 32 (w mod 4) ..), warps 2-3 idle.
// Tensor memory (512 columns): S_A, S_B, O_A, O_B.  Every wait is bounded (sm100::mbar_wait).
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tmap.h"

namespace msa {
namespace {

constexpr int kTile = 128 * 128 * 2;  // one 128-row x 128 bf16 tile (two SW128 panels)
constexpr int kDRing = 4;             // K / V ring slots (loads alternate K, V)
constexpr int kDStage = 32 * 64;      // epilogue staging per warp: 32 rows x 64 bytes
constexpr int kUR = 4;                // work-unit ring
constexpr float kRescale = 8.f;       // log2 of the largest P kept without moving the row max

struct DenseArgs {
  Dims d;
  bf16* o;
  float* lse;
  unsigned* status;
  int* sched;  // work-unit counter (zero at launch)
  int npairs;  // tile pairs per query block (G / 2, at least 1)
};

struct DenseShared {
  int u_ring[kUR];
  uint64_t q_full, q_empty, kv_full[kDRing], kv_empty[kDRing], s_full[2], p_full[2], o_full[2],
      o_free[2], u_full[kUR], u_empty[kUR], mma_done;
  uint32_t tmem;
};

__device__ __forceinline__ uint32_t par(long long k) { return (uint32_t)(k & 1); }
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Unit {
  int b, g, m, tA;  // tile A starts at token m * 128 + tA; tile B (if any) TT tokens later
  bool hasB;
};
template <int G>
__device__ __forceinline__ Unit decode_unit(const Dims& d, int npairs, int u) {
  constexpr int TT = 128 / G;
  const int per_m = d.B * d.Hkv * npairs;
  Unit x;
  x.m = d.nblk - 1 - u / per_m;  // longest units first
  const int rem = u % per_m;
  const int bg = rem / npairs, pr = rem % npairs;
  x.b = bg / d.Hkv;
  x.g = bg % d.Hkv;
  x.tA = 2 * pr * TT;
  x.hasB = G >= 2;
  return x;
}

}  // namespace

template <int G>
__global__ void __launch_bounds__(384, 1)
    dense_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, DenseArgs A) {
  using namespace sm100;
  constexpr int TT = 128 / G;  // tokens per tile
  const Dims& d = A.d;
  extern __shared__ uint8_t smem_raw[];
  DenseShared* sh = reinterpret_cast<DenseShared*>(smem_raw);
  uint8_t* base = align1024(smem_raw + sizeof(DenseShared));
  uint8_t* sQ = base;                    // [2 tiles][128 rows][128 d]  (TMA)
  uint8_t* sR = sQ + 2 * kTile;          // K / V ring [kDRing][128 keys][128 d]  (TMA)
  uint8_t* sSt = sR + kDRing * kTile;    // epilogue staging [8 warps][32 rows][64 bytes]
  const uint32_t aQ = smem_u32(sQ), aR = smem_u32(sR), aSt = smem_u32(sSt);
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const float sl2 = d.scale * kLog2e;
  const long long total = (long long)d.nblk * d.B * d.Hkv * A.npairs;

  if (tid == 0) {
    mbar_init(&sh->q_full, 1);
    mbar_init(&sh->q_empty, 1);
    for (int x = 0; x < kDRing; ++x) {
      mbar_init(&sh->kv_full[x], 1);
      mbar_init(&sh->kv_empty[x], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sh->s_full[x], 1);
      mbar_init(&sh->p_full[x], 4);
      mbar_init(&sh->o_full[x], 1);
      mbar_init(&sh->o_free[x], 4);
    }
    for (int x = 0; x < kUR; ++x) {
      mbar_init(&sh->u_full[x], 1);
      mbar_init(&sh->u_empty[x], 9);  // MMA warp, 8 softmax warps
    }
    mbar_init(&sh->mma_done, 1);
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
  const uint32_t S0 = tmem, O0 = tmem + 256;  // S_X = S0 + 128 X, O_X = O0 + 128 X
  bool ok = true;
  // unit number ni of this block, for a whole warp (published by warp 0 from a shared counter)
  auto take_unit = [&](long long ni, int& v) -> bool {
    const int x = (int)(ni % kUR);
    if (!mbar_wait_warp(&sh->u_full[x], par(ni / kUR), A.status)) return false;
    v = sh->u_ring[x];
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh->u_empty[x]);
    return true;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- units + TMA
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    long long nl = 0, pub = 0;  // K / V loads issued, unit numbers published
    bool last = false;
    for (long long ni = 0; ok; ++ni) {
      while (!last && pub < ni + 2) {  // unit numbers up to two units ahead of the loads
        const int x = (int)(pub % kUR);
        if (pub >= kUR && !mbar_wait_warp(&sh->u_empty[x], par(pub / kUR - 1), A.status)) {
          ok = false;
          break;
        }
        int v = 0;
        if (lane == 0) {
          v = atomicAdd(A.sched, 1);
          sh->u_ring[x] = v;
          mbar_arrive(&sh->u_full[x]);
        }
        v = __shfl_sync(0xffffffffu, v, 0);
        last = v >= total;
        ++pub;
      }
      if (!ok) break;
      int u = 0;
      if (lane == 0) u = sh->u_ring[ni % kUR];
      u = __shfl_sync(0xffffffffu, u, 0);
      if (u >= total) break;
      const Unit un = decode_unit<G>(d, A.npairs, u);
      const int row0 = un.b * d.S;
      // query tiles of this unit, once the previous unit's S products have read theirs
      if (ni > 0 && !mbar_wait_warp(&sh->q_empty, par(ni - 1), A.status)) { ok = false; break; }
      if (lane == 0) {
        const int t0 = un.m * kBlock + un.tA;
        mbar_expect_tx(&sh->q_full, (un.hasB ? 2 : 1) * kTile);
        tma_load_3d(sQ, &tm_q, 0, un.g * G, row0 + t0, &sh->q_full);
        tma_load_3d(sQ + kTile / 2, &tm_q, 64, un.g * G, row0 + t0, &sh->q_full);
        if (un.hasB) {
          tma_load_3d(sQ + kTile, &tm_q, 0, un.g * G, row0 + t0 + TT, &sh->q_full);
          tma_load_3d(sQ + kTile + kTile / 2, &tm_q, 64, un.g * G, row0 + t0 + TT, &sh->q_full);
        }
      }
      __syncwarp();
      for (int n = 0; n <= un.m && ok; ++n) {
        for (int w = 0; w < 2; ++w, ++nl) {  // K_n, then V_n
          const int slot = (int)(nl % kDRing);
          const long long use = nl / kDRing;
          if (use >= 1 && !mbar_wait_warp(&sh->kv_empty[slot], par(use - 1), A.status)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            uint8_t* dst = sR + slot * kTile;
            const CUtensorMap* tm = w == 0 ? &tm_k : &tm_v;
            mbar_expect_tx(&sh->kv_full[slot], kTile);
            tma_load_3d(dst, tm, 0, un.g, row0 + n * kBlock, &sh->kv_full[slot]);
            tma_load_3d(dst + kTile / 2, tm, 64, un.g, row0 + n * kBlock, &sh->kv_full[slot]);
          }
          __syncwarp();
        }
      }
    }
    // no copy may still be landing in shared memory when the block exits
    for (long long x = (nl >= kDRing ? nl - kDRing : 0); x < nl; ++x)
      mbar_wait_warp(&sh->kv_full[x % kDRing], par(x / kDRing), A.status);
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t id_s = idesc_bf16(128, 128, false, false);  // S = Q K^T
    constexpr uint32_t id_o = idesc_bf16(128, 128, false, true);   // O += P V
    long long nl = 0;               // K / V loads consumed (same sequence as the producer)
    long long cs[2] = {0, 0};       // S products issued per tile (s_full / p_full phases)
    long long nu = 0;               // units done by this block
    // O_X += P_X V for the S product number j of tile X (the unit's block n), V in ring slot vs
    auto mma_o = [&](int X, long long j, bool first, int vslot, long long vuse, bool last_of_unit,
                     bool free_v) -> bool {
      if (!mbar_wait_warp(&sh->p_full[X], par(j), A.status)) return false;
      if (first && nu > 0 && !mbar_wait_warp(&sh->o_free[X], par(nu - 1), A.status)) return false;
      if (X == 0 && !mbar_wait_warp(&sh->kv_full[vslot], par(vuse), A.status)) return false;
      fence_after_sync();
      if (lane == 0) {
        const uint32_t aV = aR + vslot * kTile;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ts(O0 + 128 * X, S0 + 128 * X + ks * 8, desc_mnmajor(aV, 128, ks), id_o, !first || ks > 0);
        if (last_of_unit) mma_commit(&sh->o_full[X]);
        if (free_v) mma_commit(&sh->kv_empty[vslot]);
      }
      __syncwarp();
      return true;
    };
    auto mma_s = [&](int X, int kslot, bool free_k, bool free_q) {
      fence_after_sync();
      if (lane == 0) {
        const uint32_t aQx = aQ + X * kTile, aK = aR + kslot * kTile;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ss(S0 + 128 * X, desc_kmajor(aQx, 128, ks), desc_kmajor(aK, 128, ks), id_s, ks > 0);
        mma_commit(&sh->s_full[X]);
        if (free_k) mma_commit(&sh->kv_empty[kslot]);
        if (free_q) mma_commit(&sh->q_empty);
      }
      __syncwarp();
    };
    for (long long ni = 0; ok; ++ni) {
      int u;
      if (!take_unit(ni, u)) { ok = false; break; }
      if (u >= total) break;
      const Unit un = decode_unit<G>(d, A.npairs, u);
      if (!mbar_wait_warp(&sh->q_full, par(nu), A.status)) { ok = false; break; }
      int pv_slot = 0;  // ring slot of V_{n-1}
      long long pv_use = 0;
      for (int n = 0; n <= un.m; ++n) {
        const int kslot = (int)(nl % kDRing);
        const long long kuse = nl / kDRing;
        const int vslot = (int)((nl + 1) % kDRing);
        const long long vuse = (nl + 1) / kDRing;
        nl += 2;
        if (!mbar_wait_warp(&sh->kv_full[kslot], par(kuse), A.status)) { ok = false; break; }
        const bool lastn = n == un.m;
        // tile A: O_A(n-1), then S_A(n)
        if (n > 0 && !mma_o(0, cs[0] - 1, n == 1, pv_slot, pv_use, false, !un.hasB)) { ok = false; break; }
        mma_s(0, kslot, !un.hasB, lastn && !un.hasB);
        ++cs[0];
        if (un.hasB) {
          if (n > 0 && !mma_o(1, cs[1] - 1, n == 1, pv_slot, pv_use, false, true)) { ok = false; break; }
          mma_s(1, kslot, true, lastn);
          ++cs[1];
        }
        pv_slot = vslot;
        pv_use = vuse;
      }
      if (!ok) break;
      // the last block's O products
      if (!mma_o(0, cs[0] - 1, un.m == 0, pv_slot, pv_use, true, !un.hasB)) { ok = false; break; }
      if (un.hasB && !mma_o(1, cs[1] - 1, un.m == 0, pv_slot, pv_use, true, true)) { ok = false; break; }
      ++nu;
    }
    if (lane == 0) mma_commit(&sh->mma_done);
    __syncwarp();
    mbar_wait_warp(&sh->mma_done, 0, A.status);
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax + epilogue
    const int X = (warp - 4) >> 2;  // tile A (warps 4-7) or B (warps 8-11)
    const int w4 = warp % 4;
    const int r = w4 * 32 + lane;  // tile row = tensor-memory lane
    const uint32_t lb = static_cast<uint32_t>(w4 * 32) << 16;
    const uint32_t Sx = S0 + 128 * X + lb, Ox = O0 + 128 * X + lb;
    const uint32_t stw = aSt + (warp - 4) * kDStage;
    long long cs = 0, nu = 0;
    for (long long ni = 0; ok; ++ni) {
      int u;
      if (!take_unit(ni, u)) { ok = false; break; }
      if (u >= total) break;
      const Unit un = decode_unit<G>(d, A.npairs, u);
      if (X == 1 && !un.hasB) continue;
      const int t = un.m * kBlock + un.tA + X * TT + r / G;  // this row's token
      const int h = un.g * G + r % G;                           // and query head
      float mr = -INFINITY, l = 0.f;
      for (int n = 0; n <= un.m; ++n, ++cs) {
        const int lim = n == un.m ? t - n * kBlock : kBlock - 1;  // visible columns 0 .. lim
        __syncwarp();
        if (!mbar_wait_warp(&sh->s_full[X], par(cs), A.status)) { ok = false; break; }
        fence_after_sync();
        // tcgen05.ld / st are warp-collective: the masked path is chosen per warp
        const bool full = __all_sync(0xffffffffu, lim == kBlock - 1);
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t v0[32];
          tmem_ld32(Sx + q * 32, v0);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c)
            mx = fmaxf(mx, (full || q * 32 + c <= lim) ? __uint_as_float(v0[c]) : -INFINITY);
        }
        if (n == 0) {
          mr = mx;  // column 0 is always visible: finite
        } else {
          const bool need = (mx - mr) * sl2 > kRescale;
          if (__any_sync(0xffffffffu, need)) {  // rescale O and l of this warp's rows
            const float alpha = need ? ex2((mr - mx) * sl2) : 1.f;
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
              uint32_t v0[32];
              tmem_ld32(Ox + q * 32, v0);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c) v0[c] = __float_as_uint(__uint_as_float(v0[c]) * alpha);
              tmem_st32(Ox + q * 32, v0);
            }
            l *= alpha;
            if (need) mr = mx;
          }
        }
        const float mb = mr * sl2;
        float la = 0.f, lc = 0.f;
#pragma unroll 1  // (a full unroll makes the compiler spill)
        for (int q = 0; q < 4; ++q) {
          uint32_t v0[32];
          tmem_ld32(Sx + q * 32, v0);
          tmem_wait_ld();
          uint32_t pw[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int k0 = q * 32 + 2 * c;
            // exponentiate unconditionally, then select: no per-lane branches
            float a0 = ex2(fmaf(__uint_as_float(v0[2 * c]), sl2, -mb));
            float a1 = ex2(fmaf(__uint_as_float(v0[2 * c + 1]), sl2, -mb));
            a0 = (full || k0 <= lim) ? a0 : 0.f;
            a1 = (full || k0 + 1 <= lim) ? a1 : 0.f;
            la += a0;
            lc += a1;
            pw[c] = pack_bf16(a0, a1);
          }
          tmem_st16(Sx + q * 16, pw);
        }
        l += la + lc;
        tmem_wait_st();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->p_full[X]);
      }
      if (!ok) break;
      // ---- unit end: O / l -> bf16 rows (through the warp's staging rows: 8 rows x 64
      // contiguous bytes per store instruction), LSE
      __syncwarp();
      if (!mbar_wait_warp(&sh->o_full[X], par(nu), A.status)) { ok = false; break; }
      fence_after_sync();
      const float sc = __fdividef(1.f, l);
      const long long orow = ((long long)un.b * d.S + t) * d.Hq + h;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t v0[32];
        tmem_ld32(Ox + q * 32, v0);
        tmem_wait_ld();
        if (q == 3) {  // O_X may now take the next unit's products
          fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh->o_free[X]);
        }
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          const uint32_t w0 = pack_bf16(__uint_as_float(v0[8 * u4 + 0]) * sc, __uint_as_float(v0[8 * u4 + 1]) * sc);
          const uint32_t w1 = pack_bf16(__uint_as_float(v0[8 * u4 + 2]) * sc, __uint_as_float(v0[8 * u4 + 3]) * sc);
          const uint32_t w2 = pack_bf16(__uint_as_float(v0[8 * u4 + 4]) * sc, __uint_as_float(v0[8 * u4 + 5]) * sc);
          const uint32_t w3 = pack_bf16(__uint_as_float(v0[8 * u4 + 6]) * sc, __uint_as_float(v0[8 * u4 + 7]) * sc);
          const uint32_t a = stw + lane * 64 + (((u4 + (lane >> 1)) & 3) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(a), "r"(w0), "r"(w1),
                       "r"(w2), "r"(w3)
                       : "memory");
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int rr = j * 8 + lane / 4, c = lane % 4;
          const long long orr = __shfl_sync(0xffffffffu, orow, rr);
          uint4 v;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
                       : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                       : "r"(stw + rr * 64 + (((c + (rr >> 1)) & 3) << 4)));
          *reinterpret_cast<uint4*>(A.o + orr * kD + q * 32 + c * 8) = v;
        }
        __syncwarp();
      }
      A.lse[((long long)un.b * d.Hq + h) * d.S + t] = (mr * sl2 + __log2f(l)) * kLn2;
      ++nu;
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int G>
static void dense_fwd_g(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        const DenseArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(DenseShared) + 1024 + (2 + kDRing) * (size_t)kTile + 8 * kDStage;
  cudaFuncSetAttribute(dense_fwd_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dense_fwd_kernel<G><<<num_sms(), 384, smem, st>>>(mq, mk, mv, a);
}

bool launch_dense_fwd(const Dims& d, const void* q, const void* k, const void* v, void* o,
                      float* lse, unsigned* status, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  const uint64_t qd[3] = {128, (uint64_t)d.Hq, (uint64_t)d.B * d.S};
  const uint64_t qs[2] = {128 * 2, (uint64_t)d.Hq * 128 * 2};
  const uint32_t qb[3] = {64, (uint32_t)d.G, (uint32_t)(128 / d.G)};
  const uint64_t kvd[3] = {128, (uint64_t)d.Hkv, (uint64_t)d.B * d.S};
  const uint64_t kvs[2] = {128 * 2, (uint64_t)d.Hkv * 128 * 2};
  const uint32_t kvb[3] = {64, 1, 128};
  if (!make_tmap_bf16(&mq, q, 3, qd, qs, qb) || !make_tmap_bf16(&mk, k, 3, kvd, kvs, kvb) ||
      !make_tmap_bf16(&mv, v, 3, kvd, kvs, kvb))
    return false;
  DenseArgs a;
  a.d = d;
  a.o = (bf16*)o;
  a.lse = lse;
  a.status = status;
  a.sched = reinterpret_cast<int*>(status + kSchedDenseFwd);
  a.npairs = d.G >= 2 ? d.G / 2 : 1;
  cudaMemsetAsync(a.sched, 0, sizeof(int), st);
  switch (d.G) {
    case 1: dense_fwd_g<1>(mq, mk, mv, a, st); break;
    case 2: dense_fwd_g<2>(mq, mk, mv, a, st); break;
    case 4: dense_fwd_g<4>(mq, mk, mv, a, st); break;
    case 8: dense_fwd_g<8>(mq, mk, mv, a, st); break;
    case 16: dense_fwd_g<16>(mq, mk, mv, a, st); break;
    default: return false;
  }
  return true;
}

}  // namespace msa
