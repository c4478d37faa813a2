// Proxy scores + causal block max-pool + streaming top-k (blog, "Forward > Proxy attention";
// forum summary, "Architecture" and "Exp-free TopK").
//
// A CTA owns the 128 tokens of query block qb for one group g.  Every key block n < qb is fully
// visible to all of them (the local block qb is forced in and never scored), so the causal mask
// reduces to "stream blocks 0 .. qb-1".  For each streamed block the CTA forms the 128 x 128 raw
// score tile qp . kp (the positive scale does not change the order, so it is not applied),
// max-pools each row over the block, and inserts the block score into that row's running list of
// the best top_k - 1 non-local blocks.  Ties keep the earlier (lower) block: a new score enters
// only if strictly larger than the current last entry and is placed after equal entries.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {

__global__ void __launch_bounds__(256, 1)
    proxy_topk_kernel(Dims d, const bf16* __restrict__ qp, const bf16* __restrict__ kp,
                      int32_t* __restrict__ idx) {
  extern __shared__ __align__(128) uint8_t smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  bf16* sK = sQ + 128 * kLd;  // [2][128][kLd]
  const int KL = d.top_k - 1;  // list length (non-local picks)
  const int KLc = KL > 0 ? KL : 1;
  float* sval = reinterpret_cast<float*>(sK + 2 * 128 * kLd);  // [128][KLc]
  int* sidx = reinterpret_cast<int*>(sval + 128 * KLc);       // [128][KLc]
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int nbg = d.B * d.Hp;
  const int qb = d.nblk - 1 - blockIdx.x / nbg;  // most work first
  const int bg = blockIdx.x % nbg;
  const int b = bg / d.Hp, g = bg % d.Hp;
  const int t0 = qb * kBlock;

  load_rows_async(sQ, 128, [&](int r) -> const bf16* {
    return qp + (((size_t)b * d.S + t0 + r) * d.Hp + g) * kD;
  }, tid, 256, qp);
  auto load_block = [&](int n, int buf) {
    load_rows_async(sK + buf * 128 * kLd, 128, [&](int r) -> const bf16* {
      return kp + ((size_t)b * d.S + n * kBlock + r) * kD;
    }, tid, 256, kp);
  };
  if (qb > 0) load_block(0, 0);
  cp_async_commit();
  for (int i = tid; i < 128 * KLc; i += 256) {
    sval[i] = -INFINITY;
    sidx[i] = -1;
  }

  // Row owner: lane%4 == 0 owns row lane/4, lane%4 == 1 owns row lane/4 + 8 (of this warp).
  const int own = lane % 4;
  const int my_row = warp * 16 + lane / 4 + (own == 1 ? 8 : 0);
  float kth = -INFINITY;  // current last list entry of my row (cached)

#pragma unroll 1
  for (int n = 0; n < qb; ++n) {
    if (n + 1 < qb) {
      load_block(n + 1, (n + 1) & 1);
      cp_async_commit();
      cp_async_wait_group<1>();
    } else {
      cp_async_wait_group<0>();
    }
    __syncthreads();
    float acc[16][4];
    zero_acc(acc);
    warp_gemm_abt<128, 128>(acc, sQ + warp * 16 * kLd, kLd, sK + (n & 1) * 128 * kLd, kLd, lane);
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      m0 = fmaxf(m0, fmaxf(acc[j][0], acc[j][1]));
      m1 = fmaxf(m1, fmaxf(acc[j][2], acc[j][3]));
    }
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
    if (own < 2 && KL > 0) {
      const float c = own == 0 ? m0 : m1;
      if (c > kth) {
        float* v = sval + my_row * KLc;
        int* ix = sidx + my_row * KLc;
        int p = KL - 1;
        while (p > 0 && v[p - 1] < c) {
          v[p] = v[p - 1];
          ix[p] = ix[p - 1];
          --p;
        }
        v[p] = c;
        ix[p] = n;
        kth = v[KL - 1];
      }
    }
    __syncthreads();
  }
  __syncthreads();
  // Emit: the picked non-local blocks in ascending order, then the local block, then -1.
  if (tid < 128) {
    int* ix = sidx + tid * KLc;
    int nv = 0;
    for (int i = 0; i < KL; ++i)
      if (ix[i] >= 0) ix[nv++] = ix[i];
    for (int i = 1; i < nv; ++i) {  // insertion sort, nv <= 63
      const int x = ix[i];
      int j = i - 1;
      while (j >= 0 && ix[j] > x) {
        ix[j + 1] = ix[j];
        --j;
      }
      ix[j + 1] = x;
    }
    int32_t* out = idx + (((size_t)b * d.Hp + g) * d.S + t0 + tid) * d.top_k;
    for (int i = 0; i < nv; ++i) out[i] = ix[i];
    out[nv] = qb;
    for (int i = nv + 1; i < d.top_k; ++i) out[i] = -1;
  }
}

void launch_proxy_topk(const Dims& d, const void* qp, const void* kp, int32_t* idx,
                       cudaStream_t st) {
  const int KLc = d.top_k > 1 ? d.top_k - 1 : 1;
  const size_t smem = 3 * 128 * kLd * sizeof(bf16) + 128 * KLc * (sizeof(float) + sizeof(int));
  cudaFuncSetAttribute(proxy_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  proxy_topk_kernel<<<d.B * d.Hp * d.nblk, 256, smem, st>>>(d, (const bf16*)qp, (const bf16*)kp,
                                                            idx);
}

}  // namespace msa
