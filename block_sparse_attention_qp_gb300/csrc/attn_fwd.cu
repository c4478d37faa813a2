// Sparse main-attention forward on the tcgen05 tensor cores (blog, "Main attention"; forum
// summary, "GPU kernel co-design": KV-outer iteration with gathered queries and a two-phase
// forward).
//
// Phase 1 (attn_fwd_kernel): a work item is one 128-key block n of group g and up to 8 tiles of
// the tokens whose selection holds n (from the inverted block map); blocks take items in list
// order from a shared counter.  A tile is 128 rows: 128/G tokens x the G query heads of the
// group.  Per tile
//   S = Q K^T                       (tensor core, 128 x 128 fp32 in tensor memory)
//   P = exp(scale S - m), l = sum P  (softmax warps, thread = row; causal cut in the local block)
//   O = P V                         (tensor core, P read from tensor memory)
//   partial (t, h, slot) = O / l in bf16, and its log-sum-exp m + log l   (epilogue warps)
// Phase 2 (combine_kernel in fwd.cu) merges the <= top_k partials of every (t, h).
//
// Roles (448 threads): warp 0 TMA loads of K/V (a three-slot ring), the block's work-item numbers
// and tensor-memory ownership, warp 1 the MMA issuer, warps 2, 3, 12, 13 gather the tile's Q rows
// (three buffers), warps 4-7 and 8-11 two softmax + epilogue groups that take alternate tiles.
// Tensor memory (512 columns): S0, S1 (S, then P in place), O0, O1.
// The gather: TMA issues about one request per 70 cycles per SM whatever its size, so with 8 heads
// per group each token's rows come as one 2 KB box (its 8 heads x both 64-column panels, through a
// 4D view of Q whose panel stride is below its head stride): 16 requests per tile.  Other group
// sizes would need 32 or more boxes per tile, and there four cp.async warps (2,048 16-byte copies
// per tile) keep up better.
// The MMA issuer runs S of tile i before O of tile i-1, so the tensor pipe works on one tile while
// the softmax warps work on the next.  Every wait is bounded (see sm100::mbar_wait).
//
// kProxy = true runs the same pipeline as the sparse proxy normaliser of the backward (blog,
// "Proxy attention" and "Backward": the student's log-sum-exp over the selected tokens is
// recomputed there, not kept from the forward): rows are tokens (G = 1) of proxy head g, the ring
// holds only proxy-key blocks, each tile runs S = Qp Kp^T alone (no V, no O), and the softmax
// warps write the natural log-sum-exp of scale * S over each (token, slot)'s visible keys.
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
constexpr int kStageWarp = 32 * 64;            // epilogue staging per warp: 32 rows x 64 bytes
constexpr int kIR = 4;                         // work-item ring: item numbers for the block's roles

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
  int* sched;  // work-item counter (zero at launch): blocks take items in order as they get free
  // this pass: the items [*item_lo, *item_hi) (NULL: 0, the list's total) of the tokens
  // [pass_t0, pass_t0 + pass_tokens), whose partials are indexed from pass_t0
  const int* item_lo;
  const int* item_hi;
  int pass_t0, pass_tokens;
};

struct FwdShared {
  int tok[kQBuf][kFwdRows];     // token of each tile token (-1: none), per Q buffer
  int slot[kQBuf][kFwdRows];    // its selection slot
  int it_ring[kIR];             // item numbers taken by this block, in order (>= total: no more)
  uint64_t kv_full[kRing], kv_empty[kRing], q_full[kQBuf], q_empty[kQBuf], meta_free[kQBuf],
      s_full[2], p_full[2], o_full[2], o_free[2], mma_done, it_full[kIR], it_empty[kIR];
  uint32_t tmem;
};

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t par(long long k) { return (uint32_t)(k & 1); }

// Q tile loaded one token (8 query heads) per TMA box: per token 2 KB = [panel][8 rows][128 B],
// both panels of a token's rows together, so consecutive 8-row groups of a panel are 2 KB apart.
constexpr int kTokBox = 2 * 8 * 128;
__device__ __forceinline__ uint64_t desc_kmajor_tok(uint32_t tile_saddr, int ks) {
  const uint32_t a = tile_saddr + (uint32_t)((ks >> 2) * (kTokBox / 2) + (ks & 3) * 32);
  return sm100::make_desc(a, 16, kTokBox);
}
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, int c0, int c1, int c2,
                                            int c3, uint64_t* mbar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5}], [%6];\n" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(static_cast<uint32_t>(__cvta_generic_to_shared(mbar)))
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

template <int G, bool kProxy>
__global__ void __launch_bounds__(448, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_q, FwdArgs A) {
  using namespace sm100;
  constexpr int TT = kFwdRows / G;  // tokens per tile
  constexpr bool kTmaQ = G == 8 && !kProxy;  // Q rows by one TMA box per token (else cp.async)
  constexpr int kLoads = kProxy ? 1 : 2;  // ring loads per item: K (or Kp) and V
  const Dims& d = A.d;

  extern __shared__ uint8_t smem_raw[];
  FwdShared* sh = reinterpret_cast<FwdShared*>(smem_raw);
  uint8_t* base = align1024(smem_raw + sizeof(FwdShared));
  uint8_t* sR = base;                     // K/V ring: [kRing][128 keys][128 d]   (TMA)
  uint8_t* sQ = sR + kRing * kFwdTile;    // [kQBuf][128 rows][128 d]          (gathered)
  uint8_t* sSt = sQ + kQBuf * kFwdTile;   // epilogue staging, [8 warps][32 rows][64 bytes]
  const uint32_t aR = smem_u32(sR), aQ = smem_u32(sQ), aSt = smem_u32(sSt);

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const float sl2 = d.scale * kLog2e;
  long long total = A.item_hi ? *A.item_hi : *A.n_items;  // items of this pass end here
  if (total > A.max_items) total = A.max_items;
  const int item0 = A.item_lo ? *A.item_lo : 0;

  if (tid == 0) {
    for (int x = 0; x < kRing; ++x) {
      mbar_init(&sh->kv_full[x], 1);
      mbar_init(&sh->kv_empty[x], 1);
    }
    for (int x = 0; x < kQBuf; ++x) {
      mbar_init(&sh->q_full[x], 256);  // 4 gather warps x 32 lanes: a plain and a cp.async arrival each
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
    for (int x = 0; x < kIR; ++x) {
      mbar_init(&sh->it_full[x], 1);
      mbar_init(&sh->it_empty[x], 13);  // MMA, 4 gather warps, 8 softmax warps
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
  const uint32_t S0 = tmem, O0 = tmem + 256;  // S_b = S0 + 128 b, O_b = O0 + 128 b
  bool ok = true;
  // Item number ni of this block, for a whole warp.  Items are handed out in list order to
  // whichever block asks next, so the blocks stay within a short window of the list (the query
  // rows of one sequence chunk stay in L2) however unevenly long the items are.
  auto take_item = [&](long long ni, int& v) -> bool {
    const int x = (int)(ni % kIR);
    if (!mbar_wait_warp(&sh->it_full[x], par(ni / kIR), A.status)) return false;
    v = sh->it_ring[x];
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh->it_empty[x]);
    return true;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA: K, V per item
    // (the whole warp runs the loop and waits; lane 0 issues)
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    long long nl = 0;  // loads issued
    // item numbers are published up to two items ahead of the K / V loads
    long long pub = 0;
    bool last = false;
    for (long long ni = 0; ok; ++ni) {
      while (!last && pub < ni + 2) {
        const int x = (int)(pub % kIR);
        if (pub >= kIR && !mbar_wait_warp(&sh->it_empty[x], par(pub / kIR - 1), A.status)) {
          ok = false;
          break;
        }
        int v = 0;
        if (lane == 0) {
          v = item0 + atomicAdd(A.sched, 1);
          sh->it_ring[x] = v;
          mbar_arrive(&sh->it_full[x]);
        }
        v = __shfl_sync(0xffffffffu, v, 0);
        last = v >= total;
        ++pub;
      }
      if (!ok) break;
      int it = 0;
      if (lane == 0) it = sh->it_ring[ni % kIR];
      it = __shfl_sync(0xffffffffu, it, 0);
      if (it >= total) break;
      const Item item = A.items[it];
      const int n = item.seg % d.nblk;
      const int bg = (int)((item.seg % d.nseg()) / d.nblk);
      const int b = bg / d.Hp, g = bg % d.Hp;  // g: proxy head (selection row)
      const int row0 = b * d.S + n * kBlock;
      // KV head of the item's attention group; the proxy key head is shared by every group
      const int kvh = kProxy ? 0 : d.kv_of(g * d.R + item.sub);
      for (int w = 0; w < kLoads; ++w) {
        const RingPos rp = ring_pos(nl);
        if (rp.use >= 1 && !mbar_wait_warp(&sh->kv_empty[rp.slot], rp.parity ^ 1u, A.status)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* dst = sR + rp.slot * kFwdTile;
          const CUtensorMap* tm = w == 0 ? &tm_k : &tm_v;
          mbar_expect_tx(&sh->kv_full[rp.slot], kFwdTile);
          tma_load_3d(dst, tm, 0, kvh, row0, &sh->kv_full[rp.slot]);
          tma_load_3d(dst + kFwdTile / 2, tm, 64, kvh, row0, &sh->kv_full[rp.slot]);
        }
        __syncwarp();
        ++nl;
      }
    }
    // no copy may still be landing in shared memory when the block exits
    for (long long x = (nl >= kRing ? nl - kRing : 0); x < nl; ++x) {
      const RingPos rp = ring_pos(x);
      mbar_wait_warp(&sh->kv_full[rp.slot], rp.parity, A.status);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // (the whole warp runs the loop and waits; lane 0 issues the MMAs and commits)
    constexpr uint32_t id_s = idesc_bf16(128, 128, false, false);  // S = Q K^T
    constexpr uint32_t id_o = idesc_bf16(128, 128, false, true);   // O = P V
    // the O product of the previous tile, issued after the next tile's S product
    long long p_ti = -1;  // < 0: none pending
    int p_vslot = 0;
    uint32_t p_vpar = 0;
    bool p_first = false, p_last = false;
    auto mma_o = [=](long long ti, int vslot, uint32_t vpar, bool first, bool last) -> bool {
      const int b = (int)(ti & 1);
      if (!mbar_wait_warp(&sh->p_full[b], par(ti >> 1), A.status)) return false;
      if (first && !mbar_wait_warp(&sh->kv_full[vslot], vpar, A.status)) return false;
      if (ti >= 2 && !mbar_wait_warp(&sh->o_free[b], par((ti - 2) >> 1), A.status)) return false;
      fence_after_sync();
      if (lane == 0) {
        const uint32_t aV = aR + vslot * kFwdTile;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ts(O0 + 128 * b, S0 + 128 * b + ks * 8, desc_mnmajor(aV, 128, ks), id_o, ks > 0);
        mma_commit(&sh->o_full[b]);
        if (last) mma_commit(&sh->kv_empty[vslot]);
      }
      __syncwarp();
      return true;
    };
    long long ni = 0, i = 0;
    for (;; ++ni) {
      int it;
      if (!take_item(ni, it)) { ok = false; break; }
      if (it >= total) break;
      const Item item = A.items[it];
      const RingPos kp = ring_pos(kLoads * ni), vp = ring_pos(kLoads * ni + 1);
      if (!mbar_wait_warp(&sh->kv_full[kp.slot], kp.parity, A.status)) { ok = false; break; }
      const uint32_t aK = aR + kp.slot * kFwdTile;
      const int ntiles = (item.count + TT - 1) / TT;
      if (ntiles == 0) {  // (items are never empty)
        if (lane == 0) mma_commit(&sh->kv_empty[kp.slot]);
        if (!kProxy) {
          if (!mbar_wait_warp(&sh->kv_full[vp.slot], vp.parity, A.status)) { ok = false; break; }
          if (lane == 0) mma_commit(&sh->kv_empty[vp.slot]);
        }
      }
      for (int tl = 0; tl < ntiles; ++tl, ++i) {
        const int b = (int)(i & 1), qb = (int)(i % kQBuf);
        if (!mbar_wait_warp(&sh->q_full[qb], par(i / kQBuf), A.status)) { ok = false; break; }
        // S_b still holds P of tile i-2 until that tile's O product has completed (proxy mode: until
        // the softmax warps have read S of tile i-2)
        if (i >= 2 && !mbar_wait_warp(kProxy ? &sh->p_full[b] : &sh->o_full[b], par((i - 2) >> 1),
                                      A.status)) { ok = false; break; }
        // the Q rows were written by other threads' cp.async (generic proxy) and only tracked by
        // the barrier: order them before the tensor core's (async proxy) reads (TMA-written rows
        // need no fence; it is harmless there)
        fence_async_smem();
        fence_after_sync();
        if (lane == 0) {
          const uint32_t aQb = aQ + qb * kFwdTile;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ss(S0 + 128 * b, kTmaQ ? desc_kmajor_tok(aQb, ks) : desc_kmajor(aQb, 128, ks),
                   desc_kmajor(aK, 128, ks), id_s, ks > 0);
          mma_commit(&sh->s_full[b]);
          mma_commit(&sh->q_empty[qb]);
          if (tl == ntiles - 1) mma_commit(&sh->kv_empty[kp.slot]);
        }
        __syncwarp();
        if (kProxy) continue;
        if (p_ti >= 0 && !mma_o(p_ti, p_vslot, p_vpar, p_first, p_last)) { ok = false; break; }
        p_ti = i;
        p_vslot = vp.slot;
        p_vpar = vp.parity;
        p_first = tl == 0;
        p_last = tl == ntiles - 1;
      }
    }
    if (!kProxy && ok && p_ti >= 0) mma_o(p_ti, p_vslot, p_vpar, p_first, p_last);
    if (lane == 0) mma_commit(&sh->mma_done);
    __syncwarp();
    mbar_wait_warp(&sh->mma_done, 0, A.status);
  } else if (warp == 2 || warp == 3 || warp == 12 || warp == 13) {
    // ---------------------------------------------------------------- gather: Q rows
    // Four warps each fill 32 rows of every tile with cp.async (completion counted on q_full);
    // each warp loads the list entries of its tokens one tile ahead.
    const int gw = warp < 4 ? warp - 2 : warp - 10;  // 0..3: rows [32 gw, 32 gw + 32)
    constexpr int XT = (32 + G - 1) / G;             // tokens per gather warp (G = 1: 32)
    const int x0 = gw * 32 / G;                      // first token of this warp
    const uint64_t pol_q = l2_policy_evict_last();  // each query row is read once per selected block
    long long gni = 0;
    int it = 0;
    if (!take_item(gni, it)) ok = false;
    if (ok && it < total) {
      Item cur = A.items[it];
      int tl = 0;
      auto load_e = [=](int base, int count, int tile) -> int {
        const int pos = tile * TT + x0 + lane;
        return (lane < XT && pos < count) ? __ldg(A.entries + base + pos) : -1;
      };
      int e = load_e(cur.base, cur.count, 0);
      long long i = 0;
      while (true) {
        const int qb = (int)(i % kQBuf);
        if (i >= kQBuf && (!mbar_wait_warp(&sh->q_empty[qb], par(i / kQBuf - 1), A.status) ||
                           !mbar_wait_warp(&sh->meta_free[qb], par(i / kQBuf - 1), A.status))) {
          ok = false;
          break;
        }
        // G > 32 never happens (G <= 16), so every warp owns whole tokens
        if (lane < XT) {
          sh->tok[qb][x0 + lane] = e < 0 ? -1 : (e >> 8);
          sh->slot[qb][x0 + lane] = e < 0 ? 0 : (e & 255);
        }
        __syncwarp();
        const int bg = (int)((cur.seg % d.nseg()) / d.nblk);
        const int b = bg / d.Hp, a = (bg % d.Hp) * d.R + cur.sub;  // attention group
        uint8_t* dQb = sQ + qb * kFwdTile;
        if constexpr (kTmaQ) {
          // lane x < XT: token x0 + x, one box of its 8 heads' rows (a missing token loads token
          // 0's rows: finite values in a row no result reads)
          if (lane < XT) {
            const int t = sh->tok[qb][x0 + lane];
            mbar_expect_tx(&sh->q_full[qb], kTokBox);  // also this lane's first arrival
            tma_load_4d(dQb + (x0 + lane) * kTokBox, &tm_q, 0, a * G, 0, b * d.S + (t < 0 ? 0 : t),
                        &sh->q_full[qb]);
          } else {
            mbar_arrive(&sh->q_full[qb]);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int c = lane + 32 * k;                // 16-byte chunk of this warp's 32 rows
            const int r = 32 * gw + (c >> 4), ch = c & 15;
            const int t = sh->tok[qb][r / G];
            const uint32_t off = (ch >> 3) * (kFwdRows * 128) + sm100::sw128_chunk(r, ch & 7);
            const size_t grow = (((size_t)b * d.S + (t < 0 ? 0 : t)) * d.Hq + a * G + r % G) * kD + ch * 8;
            cp_async16_hint(dQb + off, A.q + grow, t >= 0, pol_q);
          }
          cp_async_arrive(&sh->q_full[qb]);
        }
        mbar_arrive(&sh->q_full[qb]);  // publishes tok / slot
        ++i;
        // advance: next tile of this item, or the first tile of the next item
        const int ntiles = (cur.count + TT - 1) / TT;
        if (tl + 1 < ntiles) {
          ++tl;
          e = load_e(cur.base, cur.count, tl);
        } else {
          if (!take_item(++gni, it)) { ok = false; break; }
          if (it >= total) break;
          cur = A.items[it];
          tl = 0;
          e = load_e(cur.base, cur.count, 0);
        }
      }
      cp_async_wait_all();  // nothing may land after the block exits
      if constexpr (kTmaQ) {  // nor any TMA box (the waits are bounded)
        for (long long x = (i >= kQBuf ? i - kQBuf : 0); x < i; ++x)
          mbar_wait_warp(&sh->q_full[x % kQBuf], par(x / kQBuf), A.status);
      }
    }
  } else {
    // ---------------------------------------------------------------- softmax + epilogue
    // Warps 4-7 and 8-11 form two groups that take alternate tiles (group sg owns S and O buffer
    // sg): per tile the group writes P over S, and once O = P V has landed it writes the tile's
    // partials, while the other group works on the next tile.
    const int sg = (warp - 4) >> 2;
    const int w4 = warp % 4;       // tensor-memory lane quadrant of this warp
    const int r = w4 * 32 + lane;  // tile row = tensor-memory lane
    const uint32_t lb = static_cast<uint32_t>(w4 * 32) << 16;
    const uint32_t stw = aSt + (warp - 4) * kStageWarp;  // this warp's staging: [32 rows][64 bytes]
    const uint64_t pol_part = l2_policy_evict_first();    // partials are read once, by the combine
    long long i = 0;
    for (long long ni = 0; ok; ++ni) {
      int it;
      if (!take_item(ni, it)) { ok = false; break; }
      if (it >= total) break;
      const Item item = A.items[it];
      const int n = item.seg % d.nblk;
      const int bg = (int)((item.seg % d.nseg()) / d.nblk);
      const int b = bg / d.Hp, a = (bg % d.Hp) * d.R + item.sub;  // attention group
      const int ntiles = (item.count + TT - 1) / TT;
      for (int tl = 0; tl < ntiles; ++tl, ++i) {
        const int bb = (int)(i & 1), qb = (int)(i % kQBuf);
        if (bb != sg) continue;  // the other group's tile
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
          // ---- every key of every row of this warp visible
          float mxa = -INFINITY, mxb = -INFINITY;  // two chains of three-input maxima
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t v0[32];
            tmem_ld32(Sb + q * 32, v0);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              mxa = fmax3(mxa, __uint_as_float(v0[4 * c]), __uint_as_float(v0[4 * c + 1]));
              mxb = fmax3(mxb, __uint_as_float(v0[4 * c + 2]), __uint_as_float(v0[4 * c + 3]));
            }
          }
          m2 = fmaxf(mxa, mxb) * sl2;
          // even and odd keys summed in two fp32 chains (la, lc) by packed adds
          float2 lac = make_float2(0.f, 0.f);
          const float2 sl2x2 = make_float2(sl2, sl2), nm2 = make_float2(-m2, -m2);
#pragma unroll 1  // (a full unroll makes the compiler spill)
          for (int q = 0; q < 4; ++q) {
            uint32_t v0[32];
            tmem_ld32(Sb + q * 32, v0);
            tmem_wait_ld();
            uint32_t pw[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float2 x = ffma2(make_float2(__uint_as_float(v0[2 * c]), __uint_as_float(v0[2 * c + 1])),
                                     sl2x2, nm2);
              const float a0 = ex2f(x.x), a1 = ex2f(x.y);
              lac = fadd2(lac, make_float2(a0, a1));
              pw[c] = pack_bf16(a0, a1);
            }
            if constexpr (!kProxy) tmem_st16(Sb + q * 16, pw);
          }
          l = lac.x + lac.y;
        } else {
          // ---- some row of this warp is in its local block (keys after the token masked) or is
          // a padding row (lim = -1)
          float mx = -INFINITY;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t v0[32];
            tmem_ld32(Sb + q * 32, v0);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c)
              mx = fmaxf(mx, q * 32 + c <= lim ? __uint_as_float(v0[c]) : -INFINITY);
          }
          m2 = lim < 0 ? 0.f : mx * sl2;
          // the row sum adds in the same order as on the unmasked path (masked keys add an exact
          // 0), so a row's result does not depend on which rows share its warp -- and so not on
          // the order in which the list building placed the tokens
          float2 lac = make_float2(0.f, 0.f);
          const float2 sl2x2 = make_float2(sl2, sl2), nm2 = make_float2(-m2, -m2);
#pragma unroll 1  // (a full unroll makes the compiler spill)
          for (int q = 0; q < 4; ++q) {
            uint32_t v0[32];
            tmem_ld32(Sb + q * 32, v0);
            tmem_wait_ld();
            uint32_t pw[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int k0 = q * 32 + 2 * c;
              // exponentiate unconditionally, then select: no per-lane branches
              const float2 x = ffma2(make_float2(__uint_as_float(v0[2 * c]), __uint_as_float(v0[2 * c + 1])),
                                     sl2x2, nm2);
              float a0 = ex2f(x.x), a1 = ex2f(x.y);
              a0 = k0 <= lim ? a0 : 0.f;
              a1 = k0 + 1 <= lim ? a1 : 0.f;
              lac = fadd2(lac, make_float2(a0, a1));
              pw[c] = pack_bf16(a0, a1);
            }
            if constexpr (!kProxy) tmem_st16(Sb + q * 16, pw);
          }
          l = lac.x + lac.y;
        }
        const bool valid = t >= 0;
        const long long dst =
            valid ? (((long long)b * A.pass_tokens + (t - A.pass_t0)) * d.Hq + a * G + r % G) * d.top_k + slot : -1;
        const float sc = valid ? __fdividef(1.f, l) : 0.f;
        const float lse = valid ? (m2 + __log2f(l)) * kLn2 : 0.f;
        tmem_wait_st();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->p_full[bb]);  // proxy mode: S_b read
        if constexpr (kProxy) {  // the partial log-sum-exp is all the proxy normaliser needs
          if (valid) A.lpart[dst] = lse;
          continue;
        }
        // ---- epilogue of this tile: O / l -> bf16 partials, 32 columns at a time through the
        // warp's staging rows (16-byte chunks rotated by row pair: conflict-free both ways),
        // leaving as 8 rows x 64 contiguous bytes per store instruction
        if (!mbar_wait_warp(&sh->o_full[bb], par(i >> 1), A.status)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const uint32_t Ob = O0 + 128 * bb + lb;
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          uint32_t v0[32];
          tmem_ld32(Ob + q * 32, v0);
          tmem_wait_ld();
          if (q == 3) {  // O_b may now be overwritten by the O product of tile i+2
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh->o_free[bb]);
          }
          const float2 sc2 = make_float2(sc, sc);
          auto scaled = [&](int c) -> uint32_t {  // O columns c, c+1 times 1 / l, as bf16 pair
            const float2 o2 = fmul2(make_float2(__uint_as_float(v0[c]), __uint_as_float(v0[c + 1])), sc2);
            return pack_bf16(o2.x, o2.y);
          };
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t w0 = scaled(8 * u + 0);
            const uint32_t w1 = scaled(8 * u + 2);
            const uint32_t w2 = scaled(8 * u + 4);
            const uint32_t w3 = scaled(8 * u + 6);
            const uint32_t a = stw + lane * 64 + (((u + (lane >> 1)) & 3) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(a), "r"(w0), "r"(w1),
                         "r"(w2), "r"(w3)
                         : "memory");
          }
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int rr = j * 8 + lane / 4, c = lane % 4;
            const long long drr = __shfl_sync(0xffffffffu, dst, rr);
            uint4 v;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(stw + rr * 64 + (((c + (rr >> 1)) & 3) << 4)));
            if (drr >= 0) st_global_v4_hint(A.opart + drr * kD + q * 32 + c * 8, v, pol_part);
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

template <int G, bool kProxy>
static void attn_fwd_g(const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mq,
                       const FwdArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(FwdShared) + 1024 + (kRing + kQBuf) * kFwdTile + 8 * kStageWarp;
  cudaFuncSetAttribute(attn_fwd_kernel<G, kProxy>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smem);
  attn_fwd_kernel<G, kProxy><<<num_sms(), 448, smem, st>>>(mk, mv, mq, a);
}

int fwd_item_tiles() { return kFwdItemTiles; }

// Rank-4 bf16 tensor map, 128-byte swizzle (the Q view of the 8-heads-per-group forward).
static bool make_tmap_q4(CUtensorMap* m, const void* base, const uint64_t* dims,
                         const uint64_t* strides_bytes, const uint32_t* box) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base),
                         (const cuuint64_t*)dims, (const cuuint64_t*)strides_bytes,
                         (const cuuint32_t*)box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool launch_attn_fwd(const Dims& d, const void* q, const void* k, const void* v,
                     const int* seg_offset, const int* entries, const Item* items,
                     const int* n_items, long long max_items, const int* item_lo,
                     const int* item_hi, int pass_t0, int pass_tokens, void* opart, float* lpart,
                     unsigned* status, cudaStream_t st) {
  CUtensorMap mk, mv;
  const uint64_t kvd[3] = {128, (uint64_t)d.Hkv, (uint64_t)d.B * d.S};
  const uint64_t kvs[2] = {128 * 2, (uint64_t)d.Hkv * 128 * 2};
  const uint32_t kvb[3] = {64, 1, 128};
  if (!make_tmap_bf16(&mk, k, 3, kvd, kvs, kvb) || !make_tmap_bf16(&mv, v, 3, kvd, kvs, kvb))
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
  a.sched = reinterpret_cast<int*>(status + kSchedAttnFwd);
  a.item_lo = item_lo;
  a.item_hi = item_hi;
  a.pass_t0 = pass_t0;
  a.pass_tokens = pass_tokens;
  // 8 heads per group: Q as a 4D tensor (64 columns, head, 64-column panel, token) so that one box
  // {64, 8, 2, 1} brings a token's group rows, both panels, as 2 KB of SW128 rows
  CUtensorMap mq = mk;  // (unused by the other group sizes)
  if (d.G == 8) {
    const uint64_t qd[4] = {64, (uint64_t)d.Hq, 2, (uint64_t)d.B * d.S};
    const uint64_t qs[3] = {128 * 2, 64 * 2, (uint64_t)d.Hq * 128 * 2};
    const uint32_t qb[4] = {64, 8, 2, 1};
    if (!make_tmap_q4(&mq, q, qd, qs, qb)) return false;
  }
  cudaMemsetAsync(a.sched, 0, sizeof(int), st);
  switch (d.G) {
    case 1: attn_fwd_g<1, false>(mk, mv, mq, a, st); break;
    case 2: attn_fwd_g<2, false>(mk, mv, mq, a, st); break;
    case 4: attn_fwd_g<4, false>(mk, mv, mq, a, st); break;
    case 8: attn_fwd_g<8, false>(mk, mv, mq, a, st); break;
    case 16: attn_fwd_g<16, false>(mk, mv, mq, a, st); break;
    default: return false;
  }
  return true;
}

bool launch_proxy_lse_sparse(const Dims& d, const void* qp, const void* kp, const int* seg_offset,
                             const int* entries, const Item* items, const int* n_items,
                             long long max_items, float* lpx_part, unsigned* status,
                             cudaStream_t st) {
  CUtensorMap mk;
  const uint64_t kd[3] = {128, 1, (uint64_t)d.B * d.S};
  const uint64_t ks[2] = {128 * 2, 128 * 2};
  const uint32_t kb[3] = {64, 1, 128};
  if (!make_tmap_bf16(&mk, kp, 3, kd, ks, kb)) return false;
  FwdArgs a;
  a.d = d;
  a.d.Hq = d.Hp;  // rows are the proxy heads' query rows: one per (token, group)
  a.d.G = 1;
  a.d.R = 1;
  a.q = (const bf16*)qp;
  a.seg_offset = seg_offset;
  a.entries = entries;
  a.items = items;
  a.n_items = n_items;
  a.max_items = max_items;
  a.opart = nullptr;
  a.lpart = lpx_part;
  a.status = status;
  a.sched = reinterpret_cast<int*>(status + kSchedProxyLse);
  a.item_lo = nullptr;  // one pass over every item and token
  a.item_hi = nullptr;
  a.pass_t0 = 0;
  a.pass_tokens = d.S;
  cudaMemsetAsync(a.sched, 0, sizeof(int), st);
  attn_fwd_g<1, true>(mk, mk, mk, a, st);
  return true;
}

}  // namespace msa
