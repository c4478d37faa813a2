// Decode step of MSA inference (forum summary, "GPU kernel co-design": the selection runs on raw
// scores -- softmax keeps the order -- at the deployment setting B = 128, k = 16; the blog's
// "Proxy attention" and "Main attention" define the two stages).  One new token per sequence b,
// at position t_b = seq_len[b] - 1 of its cache (its own K, V and proxy key already written there):
//   1. decode_scores_kernel: c[b, p, n] = max over the 128 keys j of block n of qp[b, p] . kp[b, j]
//      for every block n < t_b / 128 (the local block is forced and never scored): proxy-key
//      blocks by TMA, one tcgen05 product per block (keys x proxy heads), block maxima by warps.
//   2. decode_select_kernel: one warp per (b, p) keeps each lane's best top_k - 1 blocks sorted in
//      registers, then merges the lanes by repeated warp arg-max (ties to the lower block), adds the
//      local block and writes the selection ascending, padded with -1.
//   3. decode_attn_kernel: one block per (b, attention group a): the selected K / V blocks by TMA
//      (two stages), S^T and O^T of each block on the tensor core, online softmax across blocks.
// The whole step reads the proxy-key cache once and the selected K / V blocks once: it is bound by
// memory traffic; the tensor core keeps the arithmetic off its critical path.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tmap.h"

namespace msa {

// grid (ceil(nblk / kScoreBlocks), B), 128 threads.  Per CTA: kScoreBlocks consecutive key blocks
// of sequence b, loaded by TMA (the proxy-key cache rows of a block are contiguous: 32 KB), and one
// tcgen05 product per block, S^T = Kp_block Qp^T (M = 128 keys, N = NP >= Hp proxy heads, the
// rows beyond Hp zero), into tensor memory; thread = key then reads its NP scores and the warps
// reduce each head's maximum over the block.  The products are exact bf16 x bf16 in fp32, summed
// in the tensor core's order, as in the training selection kernel.
constexpr int kScoreBlocks = 3;  // 3 x 32 KB of proxy keys in flight per CTA, two CTAs per SM
constexpr int kKpBlock = kBlock * kD * 2;
template <int NP>
struct ScoreShared {
  uint64_t kv_full[kScoreBlocks], s_full[kScoreBlocks], mma_done;
  uint32_t tmem;
  float wmax[kScoreBlocks][4][NP];  // per block, warp and head: the warp's maximum
};
template <int NP>
__global__ void __launch_bounds__(128)
    decode_scores_kernel(const __grid_constant__ CUtensorMap tm_kp, Dims d, const bf16* __restrict__ qp,
                         const int32_t* __restrict__ seq_len, float* __restrict__ scores,
                         unsigned* status) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  ScoreShared<NP>* sh = reinterpret_cast<ScoreShared<NP>*>(smem_raw);
  uint8_t* sK = align1024(smem_raw + sizeof(ScoreShared<NP>));  // [kScoreBlocks][128 keys][128 d]
  uint8_t* sQ = sK + kScoreBlocks * kKpBlock;                    // [NP rows][128 d], K-major
  const int b = blockIdx.y, tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int len = seq_len[b];
  if (len < 1 || len > d.S) {
    if (tid == 0) atomicOr(status, kStatusBadIndex);
    return;
  }
  const int m = (len - 1) / kBlock;  // local block of the new token (forced, never scored)
  const int n0 = blockIdx.x * kScoreBlocks;
  const int nb = min(kScoreBlocks, m - n0);  // blocks of this CTA before the local one
  if (nb <= 0) return;
  if (tid == 0) {
    for (int x = 0; x < kScoreBlocks; ++x) {
      mbar_init(&sh->kv_full[x], 1);
      mbar_init(&sh->s_full[x], 1);
    }
    mbar_init(&sh->mma_done, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    __syncwarp();  // lane 0 initialised the barriers alone; the allocation is warp-collective
    tmem_alloc(&sh->tmem, 128);
    tmem_relinquish();
  }
  // the proxy queries as the B operand: SW128 K-major rows, rows Hp .. NP-1 zero
  for (int x = tid; x < NP * 16; x += 128) {
    const int r = x >> 4, ch = x & 15;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < d.Hp) v = *reinterpret_cast<const uint4*>(qp + ((size_t)b * d.Hp + r) * kD + ch * 8);
    *reinterpret_cast<uint4*>(sQ + (ch >> 3) * (NP * 128) + sw128_chunk(r, ch & 7)) = v;
  }
  fence_async_smem();  // generic-proxy writes before the tensor core's reads
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sh->tmem;
  if (tid == 0) {
    tma_prefetch_desc(&tm_kp);
    for (int x = 0; x < nb; ++x) {
      const int row = b * d.S + (n0 + x) * kBlock;
      mbar_expect_tx(&sh->kv_full[x], kKpBlock);
      tma_load_2d(sK + x * kKpBlock, &tm_kp, 0, row, &sh->kv_full[x]);
      tma_load_2d(sK + x * kKpBlock + kKpBlock / 2, &tm_kp, 64, row, &sh->kv_full[x]);
    }
    constexpr uint32_t id = idesc_bf16(128, NP, false, false);
    const uint32_t aQ = smem_u32(sQ);
    for (int x = 0; x < nb; ++x) {
      if (!mbar_wait(&sh->kv_full[x], 0, status)) break;
      fence_after_sync();
      const uint32_t aK = smem_u32(sK + x * kKpBlock);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_ss(tmem + x * NP, desc_kmajor(aK, 128, ks), desc_kmajor(aQ, NP, ks), id, ks > 0);
      mma_commit(&sh->s_full[x]);
    }
    mma_commit(&sh->mma_done);  // arrives once every product issued above has completed
  }
  __syncwarp();
  // thread = key (tensor-memory lane 32 warp + lane): its NP head scores, then each head's
  // maximum over the warp's 32 keys
  const uint32_t lrow = static_cast<uint32_t>(warp * 32) << 16;
  bool ok = true;
  for (int x = 0; x < nb; ++x) {
    if (!mbar_wait_warp(&sh->s_full[x], 0, status)) {
      ok = false;
      break;
    }
    fence_after_sync();
    uint32_t v[NP];
    if constexpr (NP == 16) tmem_ld16(tmem + lrow + x * NP, v);
    else tmem_ld32(tmem + lrow + x * NP, v);
    tmem_wait_ld();
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      if (p < d.Hp) {
        float mx = __uint_as_float(v[p]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane == 0) sh->wmax[x][warp][p] = mx;
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (ok && tid < d.Hp)
    for (int x = 0; x < nb; ++x)
      scores[((size_t)b * d.Hp + tid) * d.nblk + n0 + x] =
          fmaxf(fmaxf(sh->wmax[x][0][tid], sh->wmax[x][1][tid]),
                fmaxf(sh->wmax[x][2][tid], sh->wmax[x][3][tid]));
  if (warp == 0) {
    // no product may still write tensor memory, and no copy may still land in shared memory,
    // when the block exits
    mbar_wait_warp(&sh->mma_done, 0, status);
    for (int x = 0; x < nb; ++x) mbar_wait_warp(&sh->kv_full[x], 0, status);
    tmem_dealloc(tmem, 128);
  }
}

// One warp per (b, p); KMAX >= top_k.  Blocks n < m compete by (score desc, n asc).
template <int KMAX>
__global__ void __launch_bounds__(128)
    decode_select_kernel(Dims d, const float* __restrict__ scores, const int32_t* __restrict__ seq_len,
                         int32_t* __restrict__ block_idx) {
  const int lane = threadIdx.x % 32;
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;  // b * Hp + p
  if (row >= (long long)d.B * d.Hp) return;
  const int b = (int)(row / d.Hp);
  const int len = seq_len[b];
  if (len < 1 || len > d.S) return;  // flagged by decode_scores_kernel
  const int m = (len - 1) / kBlock;
  const int K1 = min(d.top_k - 1, m);  // non-local blocks to pick
  const float* c = scores + row * d.nblk;
  // this lane's best KMAX - 1 blocks among n = lane, lane + 32, ... (descending; ties: lower n
  // first -- the lane visits its blocks in ascending order and inserts only on strictly better)
  float vals[KMAX - 1];
  int ids[KMAX - 1];
#pragma unroll
  for (int x = 0; x < KMAX - 1; ++x) {
    vals[x] = -INFINITY;
    ids[x] = 0x7fffffff;
  }
  for (int n = lane; n < m; n += 32) {
    float cv = c[n];
    int ci = n;
    bool ins = false;
#pragma unroll
    for (int x = 0; x < KMAX - 1; ++x) {
      if (x < K1) {
        const bool take = ins || cv > vals[x] || (cv == vals[x] && ci < ids[x]);
        const float tv = vals[x];
        const int ti = ids[x];
        vals[x] = take ? cv : tv;
        ids[x] = take ? ci : ti;
        cv = take ? tv : cv;
        ci = take ? ti : ci;
        ins = take;
      }
    }
  }
  // merge: K1 rounds of warp arg-max over the lanes' list heads
  int picked = 0;  // lane 0 collects the winners
  int32_t sel[KMAX];
  for (int r = 0; r < K1; ++r) {
    float bv = vals[0];
    int bi = ids[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (ids[0] == bi) {  // the winner's lane drops its head
#pragma unroll
      for (int x = 0; x < KMAX - 2; ++x) {
        vals[x] = vals[x + 1];
        ids[x] = ids[x + 1];
      }
      vals[KMAX - 2] = -INFINITY;
      ids[KMAX - 2] = 0x7fffffff;
    }
    if (lane == 0) sel[picked++] = bi;
  }
  if (lane == 0) {
    sel[picked++] = m;
    for (int i = 1; i < picked; ++i) {  // ascending
      const int x = sel[i];
      int j = i - 1;
      while (j >= 0 && sel[j] > x) {
        sel[j + 1] = sel[j];
        --j;
      }
      sel[j + 1] = x;
    }
    int32_t* out = block_idx + row * d.top_k;
    for (int i = 0; i < d.top_k; ++i) out[i] = i < picked ? sel[i] : -1;
  }
}

// One block per (b, attention group a): the group's G <= 16 query heads against its selected
// blocks of the caches, on the tensor core.  Per selected block n (K and V by TMA, two stages):
//   S^T = K_n Q^T         (M = 128 keys, N = 16: the G heads, the rest zero)   -> tensor memory
//   thread = key: the block's maximum of each head, P = exp2(scale log2(e) S - m), row sums;
//   P (bf16, [16 heads][128 keys]) -> shared memory
//   O_n^T = V_n^T P^T     (M = 128 head dims, N = 16)                         -> tensor memory
//   thread = head dim: O += O_n^T rescaled online (flash decoding over the selected blocks).
// Warps 0-3 softmax / accumulate, warp 4 TMA, warp 5 MMA issue.  Every wait is bounded.
constexpr int kAttnThreads = 192;
constexpr int kNH = 16;                   // MMA N: heads of the group, padded
constexpr int kKVTile = kBlock * kD * 2;  // one 128 x 128 bf16 tile (32 KB)
struct AttnShared {
  uint64_t kv_full[2], kv_empty[2], s_full, p_full, o_full, mma_done;
  uint32_t tmem;
  int nsel;
  int sel[64];            // the valid selected blocks, in order
  float wred[4][kNH];     // per warp and head: block maximum, then block sum
};
__global__ void __launch_bounds__(kAttnThreads)
    decode_attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       Dims d, const bf16* __restrict__ q, const int32_t* __restrict__ seq_len,
                       const int32_t* __restrict__ block_idx, bf16* __restrict__ o,
                       float* __restrict__ lse, unsigned* status) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  AttnShared* sh = reinterpret_cast<AttnShared*>(smem_raw);
  uint8_t* sK = align1024(smem_raw + sizeof(AttnShared));  // [2 stages][128 keys][128 d]
  uint8_t* sV = sK + 2 * kKVTile;                           // [2 stages][128 keys][128 d]
  uint8_t* sQ = sV + 2 * kKVTile;                           // [16 heads][128 d], K-major
  uint8_t* sP = sQ + kNH * kD * 2;                          // [16 heads][128 keys], K-major
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int G = d.G, Ha = d.Hp * d.R;
  const int b = blockIdx.x / Ha, a = blockIdx.x % Ha;
  const int p = a / d.R, kvh = d.kv_of(a);
  const int len = seq_len[b];
  if (len < 1 || len > d.S) return;  // flagged by decode_scores_kernel
  const int t = len - 1;
  if (tid == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sh->kv_full[x], 1);
      mbar_init(&sh->kv_empty[x], 1);
    }
    mbar_init(&sh->s_full, 1);
    mbar_init(&sh->p_full, 1);
    mbar_init(&sh->o_full, 1);
    mbar_init(&sh->mma_done, 1);
    mbar_fence_init();
    const int32_t* sel = block_idx + ((size_t)b * d.Hp + p) * d.top_k;
    int c = 0;
    for (int s = 0; s < d.top_k; ++s) {
      const int n = sel[s];
      if (n >= 0 && n <= t / kBlock) sh->sel[c++] = n;  // padding (or an invalid index) skipped
    }
    sh->nsel = c;
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(&sh->tmem, 64);  // S^T: columns 0-15, O^T: 32-47
    tmem_relinquish();
  }
  // Q rows of the group's heads (rows >= G zero) and P zero-initialised, as SW128 K-major tiles
  for (int x = tid; x < kNH * 16; x += kAttnThreads) {
    const int r = x >> 4, ch = x & 15;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < G) v = *reinterpret_cast<const uint4*>(q + ((size_t)b * d.Hq + a * G + r) * kD + ch * 8);
    *reinterpret_cast<uint4*>(sQ + (ch >> 3) * (kNH * 128) + sm100::sw128_chunk(r, ch & 7)) = v;
    *reinterpret_cast<uint4*>(sP + (ch >> 3) * (kNH * 128) + sm100::sw128_chunk(r, ch & 7)) =
        make_uint4(0u, 0u, 0u, 0u);
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sh->tmem, tS = tmem, tO = tmem + 32;
  const int nsel = sh->nsel;
  if (warp == 4) {
    // ---- TMA: K and V of selected block i into stage i & 1
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      for (int i = 0; i < nsel; ++i) {
        const int st = i & 1;
        if (i >= 2 && !mbar_wait(&sh->kv_empty[st], ((i - 2) >> 1) & 1, status)) break;
        const int row = b * d.S + sh->sel[i] * kBlock;
        mbar_expect_tx(&sh->kv_full[st], 2 * kKVTile);
        tma_load_3d(sK + st * kKVTile, &tm_k, 0, kvh, row, &sh->kv_full[st]);
        tma_load_3d(sK + st * kKVTile + kKVTile / 2, &tm_k, 64, kvh, row, &sh->kv_full[st]);
        tma_load_3d(sV + st * kKVTile, &tm_v, 0, kvh, row, &sh->kv_full[st]);
        tma_load_3d(sV + st * kKVTile + kKVTile / 2, &tm_v, 64, kvh, row, &sh->kv_full[st]);
      }
      // no copy may still be landing in shared memory when the block exits
      for (int i = nsel >= 2 ? nsel - 2 : 0; i < nsel; ++i)
        mbar_wait(&sh->kv_full[i & 1], (i >> 1) & 1, status);
    }
  } else if (warp == 5) {
    // ---- MMA issue: S^T of block i + 1 goes in behind O^T of block i
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, kNH, false, false);  // S^T = K Q^T
      constexpr uint32_t id_o = idesc_bf16(128, kNH, true, false);   // O^T = V^T P^T
      const uint32_t aQ = smem_u32(sQ), aP = smem_u32(sP);
      auto issue_s = [&](int i) -> bool {
        if (!mbar_wait(&sh->kv_full[i & 1], (i >> 1) & 1, status)) return false;
        fence_after_sync();
        const uint32_t aK = smem_u32(sK + (i & 1) * kKVTile);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ss(tS, desc_kmajor(aK, 128, ks), desc_kmajor(aQ, kNH, ks), id_s, ks > 0);
        mma_commit(&sh->s_full);
        return true;
      };
      bool ok = nsel > 0 && issue_s(0);
      for (int i = 0; ok && i < nsel; ++i) {
        // the softmax has read S^T of block i and written its P (shared memory)
        if (!mbar_wait(&sh->p_full, i & 1, status)) break;
        fence_after_sync();
        const uint32_t aV = smem_u32(sV + (i & 1) * kKVTile);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ss(tO, desc_mnmajor(aV, 128, ks), desc_kmajor(aP, kNH, ks), id_o, ks > 0);
        mma_commit(&sh->o_full);
        mma_commit(&sh->kv_empty[i & 1]);  // K and V of this stage are no longer read
        if (i + 1 < nsel) ok = issue_s(i + 1);
      }
      mma_commit(&sh->mma_done);
    }
  } else {
    // ---- softmax (thread = key) and accumulation (thread = head dimension), per block
    const int kr = tid;  // key row of S^T, head dimension of O^T (tensor-memory lane)
    const uint32_t lrow = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = d.scale * kLog2e;
    float mrun[kNH], l[kNH], oacc[kNH];
#pragma unroll
    for (int h = 0; h < kNH; ++h) {
      mrun[h] = -INFINITY;
      l[h] = 0.f;
      oacc[h] = 0.f;
    }
    // The four warps pass the same named barriers in every block whatever happens: a wait that
    // gives up only clears `ok` (warp-uniform), which skips the later waits and tensor-memory
    // reads, so no warp can be left at a barrier.
    bool ok = true;
    for (int i = 0; i < nsel; ++i) {
      const int n = sh->sel[i];
      const int lim = min(kBlock - 1, t - n * kBlock);  // visible keys 0 .. lim
      if (ok) ok = mbar_wait_warp(&sh->s_full, i & 1, status);
      fence_after_sync();
      uint32_t v[kNH];
#pragma unroll
      for (int h = 0; h < kNH; ++h) v[h] = 0u;
      if (ok) {
        tmem_ld16(tS + lrow, v);
        tmem_wait_ld();
      }
      float sc[kNH];
#pragma unroll
      for (int h = 0; h < kNH; ++h) {
        sc[h] = kr <= lim ? __uint_as_float(v[h]) * sl2 : -INFINITY;
        float mx = sc[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane == 0) sh->wred[warp][h] = mx;
      }
      fence_before_sync();
      bar_sync(1, 128);
      fence_after_sync();
      float mnew[kNH], alpha[kNH];
#pragma unroll
      for (int h = 0; h < kNH; ++h) {
        const float bm = fmaxf(fmaxf(sh->wred[0][h], sh->wred[1][h]), fmaxf(sh->wred[2][h], sh->wred[3][h]));
        mnew[h] = fmaxf(mrun[h], bm);  // key 0 of every selected block is visible: finite
        alpha[h] = exp2f(mrun[h] - mnew[h]);  // 0 on the first block
        mrun[h] = mnew[h];
      }
      bar_sync(1, 128);  // every warp has read the maxima before they are overwritten by sums
      // P of this key for every head, bf16, into row h of the K-major P tile (heads >= G stay 0)
      const uint32_t prow = (uint32_t)(kr >> 6) * (kNH * 128);
#pragma unroll
      for (int h = 0; h < kNH; ++h) {
        const float pv = h < G ? exp2f(sc[h] - mnew[h]) : 0.f;  // masked keys: exp2(-inf) = 0
        *reinterpret_cast<bf16*>(sP + prow + sm100::sw128_offset(h, kr & 63)) = __float2bfloat16_rn(pv);
        float sum = pv;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lane == 0) sh->wred[warp][h] = sum;
      }
      fence_async_smem();  // P (generic-proxy stores) before the tensor core's reads
      fence_before_sync();
      bar_sync(1, 128);
      fence_after_sync();
      if (tid == 0) mbar_arrive(&sh->p_full);  // S^T read, P written
#pragma unroll
      for (int h = 0; h < kNH; ++h)
        l[h] = l[h] * alpha[h] + (sh->wred[0][h] + sh->wred[1][h] + sh->wred[2][h] + sh->wred[3][h]);
      // O += O_n^T, the running sum rescaled (thread = head dimension kr)
      if (ok) ok = mbar_wait_warp(&sh->o_full, i & 1, status);
      fence_after_sync();
      uint32_t ov[kNH];
#pragma unroll
      for (int h = 0; h < kNH; ++h) ov[h] = 0u;
      if (ok) {
        tmem_ld16(tO + lrow, ov);
        tmem_wait_ld();
      }
#pragma unroll
      for (int h = 0; h < kNH; ++h) oacc[h] = oacc[h] * alpha[h] + __uint_as_float(ov[h]);
      fence_before_sync();
      bar_sync(1, 128);  // everyone has read O^T and the sums before the next block reuses them
      fence_after_sync();
    }
    if (ok) {
#pragma unroll
      for (int h = 0; h < kNH; ++h) {
        if (h < G) {
          const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
          o[((size_t)b * d.Hq + a * G + h) * kD + kr] = __float2bfloat16_rn(oacc[h] * inv);
          if (kr == 0)
            lse[(size_t)b * d.Hq + a * G + h] = l[h] > 0.f ? (mrun[h] + log2f(l[h])) * kLn2 : -INFINITY;
        }
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) {
    mbar_wait_warp(&sh->mma_done, 0, status);  // no product may still write tensor memory
    tmem_dealloc(tmem, 64);
  }
}

bool launch_decode_scores(const Dims& d, const void* qp, const void* kp_cache,
                          const int32_t* seq_len, float* scores, unsigned* status,
                          cudaStream_t st) {
  CUtensorMap mkp;  // the proxy-key cache as rows of 128: box = one 64-column panel of a block
  const uint64_t kpd[2] = {128, (uint64_t)d.B * d.S};
  const uint64_t kps[1] = {128 * 2};
  const uint32_t kpb[2] = {64, 128};
  if (!make_tmap_bf16(&mkp, kp_cache, 2, kpd, kps, kpb)) return false;
  const dim3 g1((d.nblk + kScoreBlocks - 1) / kScoreBlocks, d.B);
#define MSA_SC(NP)                                                                               \
  {                                                                                              \
    const size_t sm = sizeof(ScoreShared<NP>) + 1024 + kScoreBlocks * (size_t)kKpBlock + NP * 256; \
    cudaFuncSetAttribute(decode_scores_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,   \
                         (int)sm);                                                               \
    decode_scores_kernel<NP><<<g1, 128, sm, st>>>(mkp, d, (const bf16*)qp, seq_len, scores,      \
                                                  status);                                       \
  }
  if (d.Hp <= 16) MSA_SC(16)
  else MSA_SC(32)
#undef MSA_SC
  return true;
}

void launch_decode_select(const Dims& d, const float* scores, const int32_t* seq_len,
                          int32_t* block_idx, cudaStream_t st) {
  const long long rows = (long long)d.B * d.Hp;
  const int g2 = (int)((rows * 32 + 127) / 128);
  if (d.top_k <= 8)
    decode_select_kernel<8><<<g2, 128, 0, st>>>(d, scores, seq_len, block_idx);
  else if (d.top_k <= 16)
    decode_select_kernel<16><<<g2, 128, 0, st>>>(d, scores, seq_len, block_idx);
  else if (d.top_k <= 32)
    decode_select_kernel<32><<<g2, 128, 0, st>>>(d, scores, seq_len, block_idx);
  else
    decode_select_kernel<64><<<g2, 128, 0, st>>>(d, scores, seq_len, block_idx);
}

bool launch_decode_attn(const Dims& d, const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* seq_len, const int32_t* block_idx, void* o, float* lse,
                        unsigned* status, cudaStream_t st) {
  CUtensorMap mk, mv;  // the caches as [B S][Hkv][128]: box = one 64-column panel of a block
  const uint64_t kvd[3] = {128, (uint64_t)d.Hkv, (uint64_t)d.B * d.S};
  const uint64_t kvs[2] = {128 * 2, (uint64_t)d.Hkv * 128 * 2};
  const uint32_t kvb[3] = {64, 1, 128};
  if (!make_tmap_bf16(&mk, k_cache, 3, kvd, kvs, kvb) || !make_tmap_bf16(&mv, v_cache, 3, kvd, kvs, kvb))
    return false;
  const size_t sm = sizeof(AttnShared) + 1024 + 4 * (size_t)kKVTile + 2 * (size_t)kNH * kD * 2;
  cudaFuncSetAttribute(decode_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  decode_attn_kernel<<<d.B * d.Hp * d.R, kAttnThreads, sm, st>>>(mk, mv, d, (const bf16*)q, seq_len,
                                                                 block_idx, (bf16*)o, lse, status);
  return true;
}

}  // namespace msa
