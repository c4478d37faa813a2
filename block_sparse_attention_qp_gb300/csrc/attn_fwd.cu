// Sparse main-attention forward on the tcgen05 tensor cores (blog, "Main attention"; forum
// summary, "GPU kernel co-design": KV-outer iteration with gathered queries and a two-phase
// forward).
//
// Phase 1 (attn_fwd_kernel): a work item is one 128-key block n of group g and up to 8 tiles of
// the tokens whose selection holds n (from the inverted block map).  A tile is 128 rows: 128/G
// tokens x the G query heads of the group.  Per tile
//   S = Q K^T                       (tensor core, 128 x 128 fp32 in tensor memory)
//   P = exp(scale S - m), l = sum P  (softmax warps, thread = row; causal cut in the local block)
//   O = P V                         (tensor core, P read from tensor memory)
//   partial (t, h, slot) = O / l in bf16, and its log-sum-exp m + log l   (epilogue warps)
// Phase 2 (combine_kernel in fwd.cu) merges the <= top_k partials of every (t, h).
//
// Roles (384 threads): warp 0 TMA loads of K/V (a three-slot ring) and tensor-memory ownership,
// warp 1 the MMA issuer, warp 2 gathers the tile's Q rows (four-row TMA gathers, three buffers),
// warp 3 idle, warps 4-7 softmax, warps 8-11 epilogue.  Tensor memory (512 columns): S0, S1 (S, then P in place), O0, O1.
// The MMA issuer runs S of tile i before O of tile i-1, so the tensor pipe works on one tile while
// the softmax warps work on the next.  Every wait is bounded (see sm100::mbar_wait).
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tmap.h"

namespace msa {
namespace {

constexpr int kFwdRows = 128;                  // rows (tokens x heads) per tile
constexpr int kFwdTile = kFwdRows * 128 * 2;   // one 128-row x 128 bf16 tile (two SW128 panels)
constexpr int kFwdItemTiles = 8;               // tiles per work item
constexpr int kRing = 3;                       // K/V ring slots (one 128 x 128 tile each)
constexpr int kQBuf = 3;                       // gathered Q buffers
constexpr int kStageWarp = 32 * 128;           // epilogue staging per warp: 32 rows x 128 bytes

struct FwdArgs {
  Dims d;
  const bf16* q;
  const int* seg_offset;
  const int* entries;
  const Item* items;
  const int* n_items;
  long long max_items;
  bf16* opart;
  float* lpart;
  unsigned* status;
};

struct FwdShared {
  int tok[kQBuf][kFwdRows];     // token of each tile token (-1: none), per Q buffer
  int slot[kQBuf][kFwdRows];    // its selection slot
  long long dst[2][kFwdRows];   // partial row (t, h, slot) of each tile row (-1: none), per O buffer
  float inv_l[2][kFwdRows];     // 1 / l of each row
  float lse[2][kFwdRows];       // natural log-sum-exp of each row's partial
  uint64_t kv_full[kRing], kv_empty[kRing], q_full[kQBuf], q_empty[kQBuf], meta_free[kQBuf],
      s_full[2], p_full[2], o_full[2], o_free[2], mma_done;
  uint32_t tmem;
};

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t par(long long k) { return (uint32_t)(k & 1); }
// Arrive on `mbar` once every cp.async this thread issued so far has landed (counts as one of
// the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint64_t* mbar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(mbar))
               : "memory");
}

// The K/V ring: loads alternate K, V, K, V, ... (load L = 2 * item + {0: K, 1: V}) over kRing
// slots, so the next item's V can land as soon as the current item's K is no longer needed.
struct RingPos {
  int slot;
  uint32_t parity;  // phase parity of this use of the slot
  long long use;    // how many times the slot was used before
};
__device__ __forceinline__ RingPos ring_pos(long long load) {
  return RingPos{(int)(load % kRing), (uint32_t)((load / kRing) & 1), load / kRing};
}

}  // namespace

template <int G>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_q, FwdArgs A) {
  using namespace sm100;
  constexpr int TT = kFwdRows / G;  // tokens per tile
  const Dims& d = A.d;

  extern __shared__ uint8_t smem_raw[];
  FwdShared* sh = reinterpret_cast<FwdShared*>(smem_raw);
  uint8_t* base = align1024(smem_raw + sizeof(FwdShared));
  uint8_t* sR = base;                     // K/V ring: [kRing][128 keys][128 d]   (TMA)
  uint8_t* sQ = sR + kRing * kFwdTile;    // [kQBuf][128 rows][128 d]          (gathered)
  uint8_t* sSt = sQ + kQBuf * kFwdTile;   // epilogue staging, [4 warps][32 rows][128 bytes]
  const uint32_t aR = smem_u32(sR), aQ = smem_u32(sQ), aSt = smem_u32(sSt);

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const float sl2 = d.scale * kLog2e;
  long long total = *A.n_items;
  if (total > A.max_items) total = A.max_items;

  if (tid == 0) {
    for (int x = 0; x < kRing; ++x) {
      mbar_init(&sh->kv_full[x], 1);
      mbar_init(&sh->kv_empty[x], 1);
    }
    for (int x = 0; x < kQBuf; ++x) {
      mbar_init(&sh->q_full[x], 1);  // the gather's expect-tx arrival; the bytes complete it
      mbar_init(&sh->q_empty[x], 1);
      mbar_init(&sh->meta_free[x], 4);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sh->s_full[x], 1);
      mbar_init(&sh->p_full[x], 4);
      mbar_init(&sh->o_full[x], 1);
      mbar_init(&sh->o_free[x], 4);
    }
    mbar_init(&sh->mma_done, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&sh->tmem, 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sh->tmem;
  const uint32_t S0 = tmem, O0 = tmem + 256;  // S_b = S0 + 128 b, O_b = O0 + 128 b
  bool ok = true;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA: K, V per item
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      long long nl = 0;  // loads issued
      for (long long it = blockIdx.x; ok && it < total; it += gridDim.x) {
        const Item item = A.items[it];
        const int n = item.seg % d.nblk;
        const int bg = (int)((item.seg % d.nseg()) / d.nblk);
        const int b = bg / d.Hp, g = bg % d.Hp;
        const int row0 = b * d.S + n * kBlock;
        for (int w = 0; w < 2; ++w) {
          const RingPos rp = ring_pos(nl);
          if (rp.use >= 1 && !mbar_wait(&sh->kv_empty[rp.slot], rp.parity ^ 1u, A.status)) {
            ok = false;
            break;
          }
          uint8_t* dst = sR + rp.slot * kFwdTile;
          const CUtensorMap* tm = w == 0 ? &tm_k : &tm_v;
          mbar_expect_tx(&sh->kv_full[rp.slot], kFwdTile);
          tma_load_3d(dst, tm, 0, g, row0, &sh->kv_full[rp.slot]);
          tma_load_3d(dst + kFwdTile / 2, tm, 64, g, row0, &sh->kv_full[rp.slot]);
          ++nl;
        }
      }
      // no copy may still be landing in shared memory when the block exits
      for (long long x = (nl >= kRing ? nl - kRing : 0); x < nl; ++x) {
        const RingPos rp = ring_pos(x);
        mbar_wait(&sh->kv_full[rp.slot], rp.parity, A.status);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, 128, false, false);  // S = Q K^T
      constexpr uint32_t id_o = idesc_bf16(128, 128, false, true);   // O = P V
      struct Pending {
        long long ti;
        RingPos v;
        bool first, last;
      };
      Pending pd{};
      bool pending = false;
      auto mma_o = [&](const Pending& p) -> bool {
        const int b = (int)(p.ti & 1);
        if (!mbar_wait(&sh->p_full[b], par(p.ti >> 1), A.status)) return false;
        if (p.first && !mbar_wait(&sh->kv_full[p.v.slot], p.v.parity, A.status)) return false;
        if (p.ti >= 2 && !mbar_wait(&sh->o_free[b], par((p.ti - 2) >> 1), A.status)) return false;
        fence_after_sync();
        const uint32_t aV = aR + p.v.slot * kFwdTile;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ts(O0 + 128 * b, S0 + 128 * b + ks * 8, desc_mnmajor(aV, 128, ks), id_o, ks > 0);
        mma_commit(&sh->o_full[b]);
        if (p.last) mma_commit(&sh->kv_empty[p.v.slot]);
        return true;
      };
      long long ni = 0, i = 0;
      for (long long it = blockIdx.x; ok && it < total; it += gridDim.x, ++ni) {
        const Item item = A.items[it];
        const RingPos kp = ring_pos(2 * ni), vp = ring_pos(2 * ni + 1);
        if (!mbar_wait(&sh->kv_full[kp.slot], kp.parity, A.status)) { ok = false; break; }
        const uint32_t aK = aR + kp.slot * kFwdTile;
        const int ntiles = (item.count + TT - 1) / TT;
        if (ntiles == 0) {  // (items are never empty)
          mma_commit(&sh->kv_empty[kp.slot]);
          if (!mbar_wait(&sh->kv_full[vp.slot], vp.parity, A.status)) { ok = false; break; }
          mma_commit(&sh->kv_empty[vp.slot]);
        }
        for (int tl = 0; tl < ntiles; ++tl, ++i) {
          const int b = (int)(i & 1), qb = (int)(i % kQBuf);
          if (!mbar_wait(&sh->q_full[qb], par(i / kQBuf), A.status)) { ok = false; break; }
          // S_b still holds P of tile i-2 until that tile's O product has completed
          if (i >= 2 && !mbar_wait(&sh->o_full[b], par((i - 2) >> 1), A.status)) { ok = false; break; }
          fence_after_sync();
          const uint32_t aQb = aQ + qb * kFwdTile;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ss(S0 + 128 * b, desc_kmajor(aQb, 128, ks), desc_kmajor(aK, 128, ks), id_s, ks > 0);
          mma_commit(&sh->s_full[b]);
          mma_commit(&sh->q_empty[qb]);
          if (tl == ntiles - 1) mma_commit(&sh->kv_empty[kp.slot]);
          if (pending && !mma_o(pd)) { ok = false; break; }
          pending = true;
          pd = Pending{i, vp, tl == 0, tl == ntiles - 1};
        }
      }
      if (ok && pending) mma_o(pd);
      mma_commit(&sh->mma_done);
      mbar_wait(&sh->mma_done, 0, A.status);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- gather: Q rows (TMA)
    // Lane j fetches rows 4j .. 4j+3 of every tile with one four-row TMA gather per 64-column
    // panel; completion is counted in bytes on q_full.  The list entries of the next tile and the
    // next work item are loaded one step ahead.
    const uint64_t pol_q = l2_policy_evict_last();  // each query row is read once per selected block
    constexpr int XL = (TT + 31) / 32;               // tile tokens per lane
    long long it = blockIdx.x;
    if (lane == 0) tma_prefetch_desc(&tm_q);
    if (it < total) {
      Item cur = A.items[it];
      long long nit = it + gridDim.x;
      Item nxt = nit < total ? A.items[nit] : cur;
      int tl = 0;
      int e[XL];
      auto load_e = [&](const Item& item, int tile) {
#pragma unroll
        for (int u = 0; u < XL; ++u) {
          const int x = lane + 32 * u;
          const int pos = tile * TT + x;
          e[u] = (x < TT && pos < item.count) ? __ldg(A.entries + item.base + pos) : -1;
        }
      };
      load_e(cur, 0);
      long long i = 0;
      while (true) {
        const int qb = (int)(i % kQBuf);
        if (i >= kQBuf && (!mbar_wait_warp(&sh->q_empty[qb], par(i / kQBuf - 1), A.status) ||
                           !mbar_wait_warp(&sh->meta_free[qb], par(i / kQBuf - 1), A.status))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int u = 0; u < XL; ++u) {
          const int x = lane + 32 * u;
          if (x < TT) {
            sh->tok[qb][x] = e[u] < 0 ? -1 : (e[u] >> 8);
            sh->slot[qb][x] = e[u] < 0 ? 0 : (e[u] & 255);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_expect_tx(&sh->q_full[qb], kFwdTile);  // publishes tok / slot
        __syncwarp();
        const int bg = (int)((cur.seg % d.nseg()) / d.nblk);
        const int b = bg / d.Hp, g = bg % d.Hp;
        int rows[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int r = 4 * lane + u;
          const int t = sh->tok[qb][r / G];
          // a padding row reads row 0 (finite data; its results are never used)
          rows[u] = t < 0 ? 0 : (int)(((long long)b * d.S + t) * d.Hq + g * G + r % G);
        }
        uint8_t* dQb = sQ + qb * kFwdTile + lane * 4 * 128;
        tma_gather4(dQb, &tm_q, 0, rows[0], rows[1], rows[2], rows[3], &sh->q_full[qb], pol_q);
        tma_gather4(dQb + kFwdTile / 2, &tm_q, 64, rows[0], rows[1], rows[2], rows[3],
                    &sh->q_full[qb], pol_q);
        ++i;
        // advance: next tile of this item, or the first tile of the next item
        const int ntiles = (cur.count + TT - 1) / TT;
        if (tl + 1 < ntiles) {
          ++tl;
          load_e(cur, tl);
        } else {
          it = nit;
          if (it >= total) break;
          cur = nxt;
          tl = 0;
          load_e(cur, 0);
          nit = it + gridDim.x;
          if (nit < total) nxt = A.items[nit];
        }
      }
      // no copy may still be landing in shared memory when the block exits
      for (long long x = (i >= kQBuf ? i - kQBuf : 0); x < i; ++x)
        mbar_wait_warp(&sh->q_full[x % kQBuf], par(x / kQBuf), A.status);
    }
  } else if (warp == 3) {
    // idle
  } else if (warp < 8) {
    // ---------------------------------------------------------------- softmax
    const int w4 = warp - 4;
    const int r = w4 * 32 + lane;  // tile row = tensor-memory lane
    const uint32_t lb = static_cast<uint32_t>(w4 * 32) << 16;
    long long i = 0;
    for (long long it = blockIdx.x; ok && it < total; it += gridDim.x) {
      const Item item = A.items[it];
      const int n = item.seg % d.nblk;
      const int bg = (int)((item.seg % d.nseg()) / d.nblk);
      const int b = bg / d.Hp, g = bg % d.Hp;
      const int ntiles = (item.count + TT - 1) / TT;
      for (int tl = 0; tl < ntiles; ++tl, ++i) {
        const int bb = (int)(i & 1), qb = (int)(i % kQBuf);
        __syncwarp();
        if (!mbar_wait_warp(&sh->s_full[bb], par(i >> 1), A.status) ||
            !mbar_wait_warp(&sh->q_full[qb], par(i / kQBuf), A.status)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const int t = sh->tok[qb][r / G];
        const int slot = sh->slot[qb][r / G];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->meta_free[qb]);
        // visible key columns of this row: 0 .. lim (the causal cut only bites in the local block)
        const int lim = t < 0 ? -1 : min(kBlock - 1, t - n * kBlock);
        const uint32_t Sb = S0 + 128 * bb + lb;
        float l = 0.f, m2 = 0.f;
        // tcgen05.ld / st are warp-collective (.sync.aligned): the path must be uniform per warp
        if (__all_sync(0xffffffffu, lim == kBlock - 1)) {
          // ---- every key of every row of this warp visible: one tensor-memory round trip
          uint32_t v[4][32];
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld32(Sb + q * 32, v[q]);
          tmem_wait_ld();
          float mq[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            mq[q] = __uint_as_float(v[q][0]);
#pragma unroll
            for (int c = 1; c < 32; ++c) mq[q] = fmaxf(mq[q], __uint_as_float(v[q][c]));
          }
          m2 = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * sl2;
          float la = 0.f, lc = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t pw[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float a0 = ex2f(fmaf(__uint_as_float(v[q][2 * c]), sl2, -m2));
              const float a1 = ex2f(fmaf(__uint_as_float(v[q][2 * c + 1]), sl2, -m2));
              la += a0;
              lc += a1;
              pw[c] = pack_bf16(a0, a1);
            }
            tmem_st16(Sb + q * 16, pw);
          }
          l = la + lc;
        } else {
          // ---- some row of this warp is in its local block (keys after the token masked) or is
          // a padding row (lim = -1)
          float mx = -INFINITY;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t v0[32], v1[32];
            tmem_ld32(Sb + h * 64, v0);
            tmem_ld32(Sb + h * 64 + 32, v1);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              if (h * 64 + c <= lim) mx = fmaxf(mx, __uint_as_float(v0[c]));
              if (h * 64 + 32 + c <= lim) mx = fmaxf(mx, __uint_as_float(v1[c]));
            }
          }
          m2 = lim < 0 ? 0.f : mx * sl2;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t v0[32], v1[32];
            tmem_ld32(Sb + h * 64, v0);
            tmem_ld32(Sb + h * 64 + 32, v1);
            tmem_wait_ld();
            uint32_t pw0[16], pw1[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int k0 = h * 64 + 2 * c, k1 = h * 64 + 32 + 2 * c;
              const float a0 = k0 <= lim ? ex2f(fmaf(__uint_as_float(v0[2 * c]), sl2, -m2)) : 0.f;
              const float a1 = k0 + 1 <= lim ? ex2f(fmaf(__uint_as_float(v0[2 * c + 1]), sl2, -m2)) : 0.f;
              const float c0 = k1 <= lim ? ex2f(fmaf(__uint_as_float(v1[2 * c]), sl2, -m2)) : 0.f;
              const float c1 = k1 + 1 <= lim ? ex2f(fmaf(__uint_as_float(v1[2 * c + 1]), sl2, -m2)) : 0.f;
              l += (a0 + a1) + (c0 + c1);
              pw0[c] = pack_bf16(a0, a1);
              pw1[c] = pack_bf16(c0, c1);
            }
            tmem_st16(Sb + h * 32, pw0);
            tmem_st16(Sb + h * 32 + 16, pw1);
          }
        }
        // row results for the epilogue (its buffer is free once the epilogue of tile i-2 read it)
        if (i >= 2 && !mbar_wait_warp(&sh->o_free[bb], par((i - 2) >> 1), A.status)) {
          ok = false;
          break;
        }
        const bool valid = t >= 0;
        sh->dst[bb][r] = valid ? (((long long)b * d.S + t) * d.Hq + g * G + r % G) * d.top_k + slot : -1;
        sh->inv_l[bb][r] = valid ? 1.f / l : 0.f;
        sh->lse[bb][r] = valid ? (m2 + log2f(l)) * kLn2 : 0.f;
        tmem_wait_st();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->p_full[bb]);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int w8 = warp - 8;
    const int r = w8 * 32 + lane;
    const uint32_t lb = static_cast<uint32_t>(w8 * 32) << 16;
    const uint32_t stw = aSt + w8 * kStageWarp;  // this warp's staging: [32 rows][128 bytes]
    const uint64_t pol_part = l2_policy_evict_first();  // partials are read once, by the combine
    long long i = 0;
    for (long long it = blockIdx.x; ok && it < total; it += gridDim.x) {
      const Item item = A.items[it];
      const int ntiles = (item.count + TT - 1) / TT;
      for (int tl = 0; tl < ntiles; ++tl, ++i) {
        const int bb = (int)(i & 1);
        __syncwarp();
        if (!mbar_wait_warp(&sh->o_full[bb], par(i >> 1), A.status) ||
            !mbar_wait_warp(&sh->p_full[bb], par(i >> 1), A.status)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const long long dst = sh->dst[bb][r];
        const float sc = sh->inv_l[bb][r];
        const float lse = sh->lse[bb][r];
        const uint32_t Ob = O0 + 128 * bb + lb;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v0[32], v1[32];
          tmem_ld32(Ob + h * 64, v0);
          tmem_ld32(Ob + h * 64 + 32, v1);
          tmem_wait_ld();
          if (h == 1) {
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh->o_free[bb]);
          }
          // this row's 64 columns -> 128 bytes of bf16 in the warp's staging (16-byte chunks
          // XOR-swizzled by row), then 4 rows x 128 contiguous bytes per store instruction
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t* src = u < 2 ? v0 : v1;
            const int o = (u & 1) * 16;
            const uint32_t w0 = pack_bf16(__uint_as_float(src[o + 0]) * sc, __uint_as_float(src[o + 1]) * sc);
            const uint32_t w1 = pack_bf16(__uint_as_float(src[o + 2]) * sc, __uint_as_float(src[o + 3]) * sc);
            const uint32_t w2 = pack_bf16(__uint_as_float(src[o + 4]) * sc, __uint_as_float(src[o + 5]) * sc);
            const uint32_t w3 = pack_bf16(__uint_as_float(src[o + 6]) * sc, __uint_as_float(src[o + 7]) * sc);
            const uint32_t w4_ = pack_bf16(__uint_as_float(src[o + 8]) * sc, __uint_as_float(src[o + 9]) * sc);
            const uint32_t w5 = pack_bf16(__uint_as_float(src[o + 10]) * sc, __uint_as_float(src[o + 11]) * sc);
            const uint32_t w6 = pack_bf16(__uint_as_float(src[o + 12]) * sc, __uint_as_float(src[o + 13]) * sc);
            const uint32_t w7 = pack_bf16(__uint_as_float(src[o + 14]) * sc, __uint_as_float(src[o + 15]) * sc);
            const uint32_t a0 = stw + lane * 128 + ((((2 * u) ^ lane) & 7) << 4);
            const uint32_t a1 = stw + lane * 128 + ((((2 * u + 1) ^ lane) & 7) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(a0), "r"(w0), "r"(w1),
                         "r"(w2), "r"(w3)
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(a1), "r"(w4_), "r"(w5),
                         "r"(w6), "r"(w7)
                         : "memory");
          }
          __syncwarp();
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int rr = u * 4 + lane / 8, c = lane % 8;
            const long long drr = __shfl_sync(0xffffffffu, dst, rr);
            uint4 v;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(stw + rr * 128 + (((c ^ rr) & 7) << 4)));
            if (drr >= 0) st_global_v4_hint(A.opart + drr * kD + h * 64 + c * 8, v, pol_part);
          }
          __syncwarp();
        }
        if (dst >= 0) A.lpart[dst] = lse;
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int G>
static void attn_fwd_g(const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mq,
                       const FwdArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(FwdShared) + 1024 + (kRing + kQBuf) * kFwdTile + 4 * kStageWarp;
  cudaFuncSetAttribute(attn_fwd_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  attn_fwd_kernel<G><<<num_sms(), 384, smem, st>>>(mk, mv, mq, a);
}

int fwd_item_tiles() { return kFwdItemTiles; }

bool launch_attn_fwd(const Dims& d, const void* q, const void* k, const void* v,
                     const int* seg_offset, const int* entries, const Item* items,
                     const int* n_items, long long max_items, void* opart, float* lpart,
                     unsigned* status, cudaStream_t st) {
  CUtensorMap mk, mv;
  const uint64_t kvd[3] = {128, (uint64_t)d.Hkv, (uint64_t)d.B * d.S};
  const uint64_t kvs[2] = {128 * 2, (uint64_t)d.Hkv * 128 * 2};
  const uint32_t kvb[3] = {64, 1, 128};
  // query rows for the four-row gathers: [B*S*Hq rows][128], box 64 columns x 1 row
  CUtensorMap mq;
  const uint64_t qd[2] = {128, (uint64_t)d.B * d.S * d.Hq};
  const uint64_t qs[1] = {128 * 2};
  const uint32_t qbx[2] = {64, 1};
  if (!make_tmap_bf16(&mk, k, 3, kvd, kvs, kvb) || !make_tmap_bf16(&mv, v, 3, kvd, kvs, kvb) ||
      !make_tmap_bf16(&mq, q, 2, qd, qs, qbx))
    return false;
  FwdArgs a;
  a.d = d;
  a.q = (const bf16*)q;
  a.seg_offset = seg_offset;
  a.entries = entries;
  a.items = items;
  a.n_items = n_items;
  a.max_items = max_items;
  a.opart = (bf16*)opart;
  a.lpart = lpart;
  a.status = status;
  switch (d.G) {
    case 1: attn_fwd_g<1>(mk, mv, mq, a, st); break;
    case 2: attn_fwd_g<2>(mk, mv, mq, a, st); break;
    case 4: attn_fwd_g<4>(mk, mv, mq, a, st); break;
    case 8: attn_fwd_g<8>(mk, mv, mq, a, st); break;
    case 16: attn_fwd_g<16>(mk, mv, mq, a, st); break;
    default: return false;
  }
  return true;
}

}  // namespace msa
