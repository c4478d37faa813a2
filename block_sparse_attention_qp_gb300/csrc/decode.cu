// Decode step of MSA inference (forum summary, "GPU kernel co-design": the selection runs on raw
// scores -- softmax keeps the order -- at the deployment setting B = 128, k = 16; the blog's
// "Proxy attention" and "Main attention" define the two stages).  One new token per sequence b,
// at position t_b = seq_len[b] - 1 of its cache (its own K, V and proxy key already written there):
//   1. decode_scores_kernel: c[b, p, n] = max over the 128 keys j of block n of qp[b, p] . kp[b, j]
//      for every block n < t_b / 128 (the local block is forced and never scored).  One thread per
//      key streams the proxy-key cache once for all Hp proxy heads.
//   2. decode_select_kernel: one warp per (b, p) keeps each lane's best top_k - 1 blocks sorted in
//      registers, then merges the lanes by repeated warp arg-max (ties to the lower block), adds the
//      local block and writes the selection ascending, padded with -1.
//   3. decode_attn_kernel: one block per (b, attention group a), one warp per query head: each
//      selected K / V block is staged in shared memory (rows padded to 272 bytes, so 16-byte reads
//      of eight rows hit distinct banks), the warp's lanes score 4 keys each, online softmax across
//      blocks, and the lanes accumulate O over 4 head-dim columns each.
// The whole step reads the proxy-key cache once and the selected K / V blocks once: it is bound by
// memory traffic, so it runs on CUDA cores.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tmap.h"

namespace msa {
namespace {

constexpr int kRow = kD + 8;  // padded bf16 row of a staged K / V block (272 bytes)

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace

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

// One block per (b, attention group a), G warps (warp = query head a G + w).
template <int G>
__global__ void __launch_bounds__(32 * G)
    decode_attn_kernel(Dims d, const bf16* __restrict__ q, const bf16* __restrict__ k_cache,
                       const bf16* __restrict__ v_cache, const int32_t* __restrict__ seq_len,
                       const int32_t* __restrict__ block_idx, bf16* __restrict__ o,
                       float* __restrict__ lse) {
  extern __shared__ __align__(16) uint8_t smem[];
  bf16* sK = reinterpret_cast<bf16*>(smem);  // [128 keys][kRow]
  bf16* sV = sK + kBlock * kRow;             // [128 keys][kRow]
  float* sP = reinterpret_cast<float*>(sV + kBlock * kRow);  // [G][128] probabilities
  const int tid = threadIdx.x, lane = tid % 32, w = tid / 32;
  const int Ha = d.Hp * d.R;
  const int b = blockIdx.x / Ha, a = blockIdx.x % Ha;
  const int p = a / d.R, kvh = d.kv_of(a), h = a * G + w;
  const int len = seq_len[b];
  if (len < 1 || len > d.S) return;  // flagged by decode_scores_kernel
  const int t = len - 1;
  const float sl2 = d.scale * kLog2e;
  // this lane's query slice: dims 4 lane .. 4 lane + 3 (for the scores, the warp reduces)
  float qv[4];
  {
    const uint2 u = *reinterpret_cast<const uint2*>(q + ((size_t)b * d.Hq + h) * kD + 4 * lane);
    qv[0] = bf_lo(u.x);
    qv[1] = bf_hi(u.x);
    qv[2] = bf_lo(u.y);
    qv[3] = bf_hi(u.y);
  }
  float mr = -INFINITY, l = 0.f, oacc[4] = {0.f, 0.f, 0.f, 0.f};
  const int32_t* sel = block_idx + ((size_t)b * d.Hp + p) * d.top_k;
  for (int s = 0; s < d.top_k; ++s) {
    const int n = sel[s];
    if (n < 0 || n > t / kBlock) continue;  // padding (or an invalid index: skipped)
    __syncthreads();  // the previous block's tiles are no longer read
    for (int x = tid; x < kBlock * 16; x += blockDim.x) {  // 16-byte chunks of 128 rows
      const int r = x >> 4, ch = x & 15;
      const size_t g = (((size_t)b * d.S + n * kBlock + r) * d.Hkv + kvh) * kD + ch * 8;
      cp_async16(sK + r * kRow + ch * 8, k_cache + g);
      cp_async16(sV + r * kRow + ch * 8, v_cache + g);
    }
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    const int lim = min(kBlock - 1, t - n * kBlock);  // visible keys 0 .. lim
    // scores: for each key, the warp's lanes hold 4 dims each and reduce across the warp;
    // lane j keeps the scores of keys j, j + 32, j + 64, j + 96
    float sc[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      sc[kk] = -INFINITY;
#pragma unroll 4
      for (int j2 = 0; j2 < 32; ++j2) {
        const int j = kk * 32 + j2;
        const uint2 u = *reinterpret_cast<const uint2*>(sK + j * kRow + 4 * lane);
        float v = qv[0] * bf_lo(u.x) + qv[1] * bf_hi(u.x) + qv[2] * bf_lo(u.y) + qv[3] * bf_hi(u.y);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (j2 == lane) sc[kk] = j <= lim ? v * sl2 : -INFINITY;
      }
    }
    float bm = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
    const float mn = fmaxf(mr, bm);  // key 0 of the local block is always visible: finite
    const float alpha = exp2f(mr - mn);  // mr = -inf on the first block: 0
    float ps = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float pv = exp2f(sc[kk] - mn);
      sP[w * kBlock + kk * 32 + lane] = pv;
      ps += pv;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
    mr = mn;
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[e] *= alpha;
    __syncwarp();
    for (int j = 0; j <= lim; ++j) {  // O += P V over this lane's 4 columns
      const float pv = sP[w * kBlock + j];
      const uint2 u = *reinterpret_cast<const uint2*>(sV + j * kRow + 4 * lane);
      oacc[0] = fmaf(pv, bf_lo(u.x), oacc[0]);
      oacc[1] = fmaf(pv, bf_hi(u.x), oacc[1]);
      oacc[2] = fmaf(pv, bf_lo(u.y), oacc[2]);
      oacc[3] = fmaf(pv, bf_hi(u.y), oacc[3]);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  *reinterpret_cast<uint2*>(o + ((size_t)b * d.Hq + h) * kD + 4 * lane) =
      make_uint2(pack_bf16(oacc[0] * inv, oacc[1] * inv), pack_bf16(oacc[2] * inv, oacc[3] * inv));
  if (lane == 0) lse[(size_t)b * d.Hq + h] = l > 0.f ? (mr + log2f(l)) * kLn2 : -INFINITY;
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

void launch_decode_attn(const Dims& d, const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* seq_len, const int32_t* block_idx, void* o, float* lse,
                        cudaStream_t st) {
  const int g3 = d.B * d.Hp * d.R;
  const size_t sm3 = 2 * (size_t)kBlock * kRow * sizeof(bf16) + (size_t)d.G * kBlock * sizeof(float);
#define MSA_DEC_CASE(GG)                                                                        \
  case GG:                                                                                      \
    cudaFuncSetAttribute(decode_attn_kernel<GG>, cudaFuncAttributeMaxDynamicSharedMemorySize,   \
                         (int)sm3);                                                             \
    decode_attn_kernel<GG><<<g3, 32 * GG, sm3, st>>>(d, (const bf16*)q, (const bf16*)k_cache,   \
                                                     (const bf16*)v_cache, seq_len, block_idx,  \
                                                     (bf16*)o, lse);                            \
    break;
  switch (d.G) {
    MSA_DEC_CASE(1)
    MSA_DEC_CASE(2)
    MSA_DEC_CASE(4)
    MSA_DEC_CASE(8)
    MSA_DEC_CASE(16)
  }
#undef MSA_DEC_CASE
}

}  // namespace msa
