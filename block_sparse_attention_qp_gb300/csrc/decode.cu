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

namespace msa {
namespace {

constexpr int kRow = kD + 8;  // padded bf16 row of a staged K / V block (272 bytes)

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace

// grid (ceil(nblk / kScoreBlocks), B), 128 threads (thread = key of the block); NP >= Hp.
constexpr int kScoreBlocks = 4;
template <int NP>
__global__ void __launch_bounds__(128)
    decode_scores_kernel(Dims d, const bf16* __restrict__ qp, const bf16* __restrict__ kp_cache,
                         const int32_t* __restrict__ seq_len, float* __restrict__ scores,
                         unsigned* status) {
  extern __shared__ float sq[];  // [Hp][128] proxy queries, then [4 warps][Hp] block maxima
  float* wmax = sq + d.Hp * kD;
  const int b = blockIdx.y, tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int len = seq_len[b];
  if (len < 1 || len > d.S) {
    if (tid == 0) atomicOr(status, kStatusBadIndex);
    return;
  }
  const int m = (len - 1) / kBlock;  // local block of the new token
  for (int x = tid; x < d.Hp * kD; x += blockDim.x) sq[x] = __bfloat162float(qp[(size_t)b * d.Hp * kD + x]);
  __syncthreads();
  for (int n = blockIdx.x * kScoreBlocks; n < min(m, (int)(blockIdx.x + 1) * kScoreBlocks); ++n) {
    const uint4* row = reinterpret_cast<const uint4*>(kp_cache + ((size_t)b * d.S + n * kBlock + tid) * kD);
    float acc[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) acc[p] = 0.f;
#pragma unroll 4
    for (int c = 0; c < 16; ++c) {
      const uint4 w = __ldg(row + c);
      const float x[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y),
                          bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        if (p < d.Hp) {
          const float* qv = sq + p * kD + c * 8;
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[p] = fmaf(qv[e], x[e], acc[p]);
        }
      }
    }
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      if (p < d.Hp) {
        float v = acc[p];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
        if (lane == 0) wmax[warp * d.Hp + p] = v;
      }
    }
    __syncthreads();
    if (tid < d.Hp)
      scores[((size_t)b * d.Hp + tid) * d.nblk + n] =
          fmaxf(fmaxf(wmax[tid], wmax[d.Hp + tid]), fmaxf(wmax[2 * d.Hp + tid], wmax[3 * d.Hp + tid]));
    __syncthreads();
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

void launch_decode(const Dims& d, const void* q, const void* qp, const void* k_cache,
                   const void* v_cache, const void* kp_cache, const int32_t* seq_len,
                   int32_t* block_idx, void* o, float* lse, float* scores, unsigned* status,
                   cudaStream_t st) {
  const dim3 g1((d.nblk + kScoreBlocks - 1) / kScoreBlocks, d.B);
  const size_t sm1 = (size_t)(d.Hp * kD + 4 * d.Hp) * sizeof(float);
#define MSA_SC(NP) decode_scores_kernel<NP><<<g1, 128, sm1, st>>>(d, (const bf16*)qp, \
                           (const bf16*)kp_cache, seq_len, scores, status)
  if (d.Hp <= 1) MSA_SC(1);
  else if (d.Hp <= 2) MSA_SC(2);
  else if (d.Hp <= 4) MSA_SC(4);
  else if (d.Hp <= 8) MSA_SC(8);
  else if (d.Hp <= 16) MSA_SC(16);
  else MSA_SC(32);
#undef MSA_SC
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
