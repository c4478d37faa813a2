// Backward: D = rowsum(dO * O), and the fused main + proxy backward (blog, "Backward" and
// "KL Divergence Loss").
//
// Fused pass.  A work item is one 64-key half of key block n of group g, plus a run of tokens that
// use the block (from the inverted block map; in warmup mode every token t >= 128 n).  The item
// keeps the half's K, V and Kp in shared memory and its dK, dV, dKp in registers while it streams
// tiles of 128/G tokens x G query heads (128 rows).  Per tile:
//   main   S = Q K^T, P = exp(scale S - LSE), dP = dO V^T, dS = P (dP - D)
//          dV += P^T dO, dK += scale dS^T Q, dQ += scale dS K        (dQ: fp32 atomics)
//   proxy  teacher  pbar = mean over the G heads of P  (detached: used as a constant)
//          student  p_px = exp(scale qp.kp - LSE_px)   (LSE_px over the same key set)
//          dz = kl_grad/(B S Hp) (p_px - pbar)          (the blog's closed form)
//          dQp += scale dz Kp (fp32 atomics), dKp += scale dz^T Qp
// dK, dV, dKp of the item are added into fp32 accumulators at the end (an item covers at most
// chunk_tiles tiles, so busy blocks are spread over several CTAs).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {

constexpr int kLdh = 72;  // padded row (bf16) of 64-column tiles

__global__ void rowdot_kernel(Dims d, const bf16* __restrict__ o, const bf16* __restrict__ dout,
                              float* __restrict__ drow) {
  const long long rows = (long long)d.B * d.S * d.Hq;
  const int lane = threadIdx.x % 32;
  for (long long r = (blockIdx.x * (long long)blockDim.x + threadIdx.x) / 32; r < rows;
       r += (long long)gridDim.x * blockDim.x / 32) {
    const uint2 a = *reinterpret_cast<const uint2*>(o + (size_t)r * kD + lane * 4);
    const uint2 c = *reinterpret_cast<const uint2*>(dout + (size_t)r * kD + lane * 4);
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* pc = reinterpret_cast<const __nv_bfloat162*>(&c);
    float s = __low2float(pa[0]) * __low2float(pc[0]) + __high2float(pa[0]) * __high2float(pc[0]) +
              __low2float(pa[1]) * __low2float(pc[1]) + __high2float(pa[1]) * __high2float(pc[1]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) {
      const int h = (int)(r % d.Hq);
      const long long bt = r / d.Hq;
      const int t = (int)(bt % d.S), b = (int)(bt / d.S);
      drow[((size_t)b * d.Hq + h) * d.S + t] = s;
    }
  }
}

struct BwdArgs {
  Dims d;
  const bf16 *q, *k, *v, *qp, *kp, *dout;
  const float *lse, *drow, *lse_px;
  float cz;  // kl_grad / (B * S * Hp)
  const int* seg_offset;
  const int* entries;
  const Item* items;
  const int* n_items;
  long long max_items;
  float *dq, *dk, *dv, *dqp, *dkp;
};

__device__ __forceinline__ void add2(float* p, float a, float b) {
  atomicAdd(reinterpret_cast<float2*>(p), make_float2(a, b));
}

template <int G, bool kDense>
__global__ void __launch_bounds__(256, 1) fused_bwd_kernel(BwdArgs A) {
  constexpr int TT = 128 / G;              // tokens per tile
  constexpr int TP = TT < 16 ? 16 : TT;    // proxy rows, padded to the 16-row product shape
  const Dims& d = A.d;
  extern __shared__ __align__(128) uint8_t smem[];
  bf16* sK = reinterpret_cast<bf16*>(smem);  // [64][kLd]
  bf16* sV = sK + 64 * kLd;
  bf16* sKp = sV + 64 * kLd;
  bf16* sQ = sKp + 64 * kLd;                 // [128][kLd]
  bf16* sdO = sQ + 128 * kLd;                // [128][kLd]
  bf16* sQp = sdO + 128 * kLd;               // [TP][kLd]
  bf16* sP = sQp + TP * kLd;                 // [128][kLdh]
  bf16* sdS = sP + 128 * kLdh;               // [128][kLdh]
  bf16* sdz = sdS + 128 * kLdh;              // [TP][kLdh]
  float* sPbar = reinterpret_cast<float*>(sdz + TP * kLdh);  // [TP][64]
  float* sLse = sPbar + TP * 64;             // [128]
  float* sD = sLse + 128;                    // [128]
  float* sLpx = sD + 128;                    // [TP]
  int* sTok = reinterpret_cast<int*>(sLpx + TP);  // [TP]

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const float sl2 = d.scale * kLog2e;
  long long total = *A.n_items;
  if (total > A.max_items) total = A.max_items;

  for (long long it = blockIdx.x; it < total; it += gridDim.x) {
    const Item item = A.items[it];
    const int n = item.seg % d.nblk;
    const int bg = item.seg / d.nblk;
    const int b = bg / d.Hp, g = bg % d.Hp;
    const int j0 = n * kBlock + item.half * 64;  // first key of the half
    load_rows_async(sK, 64, [&](int r) -> const bf16* {
      return A.k + (((size_t)b * d.S + j0 + r) * d.Hkv + g) * kD;
    }, tid, 256, A.k);
    load_rows_async(sV, 64, [&](int r) -> const bf16* {
      return A.v + (((size_t)b * d.S + j0 + r) * d.Hkv + g) * kD;
    }, tid, 256, A.v);
    load_rows_async(sKp, 64, [&](int r) -> const bf16* {
      return A.kp + ((size_t)b * d.S + j0 + r) * kD;
    }, tid, 256, A.kp);
    cp_async_commit();

    // per-item accumulators: warp w owns keys 16 (w % 4) .. +15, head-dim columns 64 (w / 4) ..
    float dv[8][4], dk[8][4], dkp[8][4];
    zero_acc(dv);
    zero_acc(dk);
    zero_acc(dkp);
    const int km0 = 16 * (warp % 4), dn0 = 64 * (warp / 4);

#pragma unroll 1
    for (int tt = 0; tt < item.count; tt += TT) {
      const int cnt = min(TT, item.count - tt);
      if (tid < TP) {
        int t = -1;
        if (tid < cnt) {
          const int pos = item.first + tt + tid;
          t = kDense ? n * kBlock + pos : (A.entries[A.seg_offset[item.seg] + pos] >> 8);
        }
        sTok[tid] = t;
      }
      __syncthreads();
      load_rows_async(sQ, 128, [&](int r) -> const bf16* {
        const int t = sTok[r / G];
        return t < 0 ? nullptr : A.q + (((size_t)b * d.S + t) * d.Hq + g * G + r % G) * kD;
      }, tid, 256, A.q);
      load_rows_async(sdO, 128, [&](int r) -> const bf16* {
        const int t = sTok[r / G];
        return t < 0 ? nullptr : A.dout + (((size_t)b * d.S + t) * d.Hq + g * G + r % G) * kD;
      }, tid, 256, A.dout);
      load_rows_async(sQp, TP, [&](int r) -> const bf16* {
        const int t = sTok[r];
        return t < 0 ? nullptr : A.qp + (((size_t)b * d.S + t) * d.Hp + g) * kD;
      }, tid, 256, A.qp);
      cp_async_commit();
      if (tid < 128) {
        const int t = sTok[tid / G];
        const size_t hrow = ((size_t)b * d.Hq + g * G + tid % G) * d.S;
        sLse[tid] = t < 0 ? 0.f : A.lse[hrow + t] * kLog2e;
        sD[tid] = t < 0 ? 0.f : A.drow[hrow + t];
      }
      if (tid < TP) {
        const int t = sTok[tid];
        sLpx[tid] = t < 0 ? 0.f : A.lse_px[((size_t)b * d.Hp + g) * d.S + t] * kLog2e;
      }
      cp_async_wait_all();
      __syncthreads();

      // ---- main probabilities and score gradients, warp rows 16 w .. 16 w + 15
      const int ra = warp * 16 + lane / 4, rb = ra + 8;
      const int ta = sTok[ra / G], tb = sTok[rb / G];
      float s[8][4], dp[8][4];
      zero_acc(s);
      zero_acc(dp);
      warp_gemm_abt<64, 128>(s, sQ + warp * 16 * kLd, kLd, sK, kLd, lane);
      warp_gemm_abt<64, 128>(dp, sdO + warp * 16 * kLd, kLd, sV, kLd, lane);
      const float la = sLse[ra], lb = sLse[rb], Da = sD[ra], Db = sD[rb];
#pragma unroll
      for (int jt = 0; jt < 8; ++jt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = j0 + 8 * jt + 2 * (lane % 4) + (e & 1);
          const int t = e < 2 ? ta : tb;
          const float p = (t >= 0 && j <= t) ? exp2f(s[jt][e] * sl2 - (e < 2 ? la : lb)) : 0.f;
          s[jt][e] = p;
          dp[jt][e] = p * (dp[jt][e] - (e < 2 ? Da : Db));
        }
      // teacher: sum the G rows of every token (rows of a token are consecutive)
#pragma unroll
      for (int jt = 0; jt < 8; ++jt) {
        float x[4] = {s[jt][0], s[jt][1], s[jt][2], s[jt][3]};
        if (G == 16) {
          x[0] += x[2];
          x[1] += x[3];
        }
#pragma unroll
        for (int off = 4; off < 4 * (G < 8 ? G : 8); off <<= 1)
#pragma unroll
          for (int e = 0; e < 4; ++e) x[e] += __shfl_xor_sync(0xffffffffu, x[e], off);
        const int col = 8 * jt + 2 * (lane % 4);
        if (G == 16) {
          if (lane / 4 == 0) {
            sPbar[warp * 64 + col] = x[0] * (1.f / G);
            sPbar[warp * 64 + col + 1] = x[1] * (1.f / G);
          }
        } else if ((lane / 4) % G == 0) {
          sPbar[(ra / G) * 64 + col] = x[0] * (1.f / G);
          sPbar[(ra / G) * 64 + col + 1] = x[1] * (1.f / G);
          sPbar[(rb / G) * 64 + col] = x[2] * (1.f / G);
          sPbar[(rb / G) * 64 + col + 1] = x[3] * (1.f / G);
        }
      }
#pragma unroll
      for (int jt = 0; jt < 8; ++jt) {
        const int col = 8 * jt + 2 * (lane % 4);
        *reinterpret_cast<uint32_t*>(sP + ra * kLdh + col) = pack_bf16(s[jt][0], s[jt][1]);
        *reinterpret_cast<uint32_t*>(sP + rb * kLdh + col) = pack_bf16(s[jt][2], s[jt][3]);
        *reinterpret_cast<uint32_t*>(sdS + ra * kLdh + col) = pack_bf16(dp[jt][0], dp[jt][1]);
        *reinterpret_cast<uint32_t*>(sdS + rb * kLdh + col) = pack_bf16(dp[jt][2], dp[jt][3]);
      }
      // dQ rows of this warp: scale dS K
      {
        uint32_t da[4][4];
        c_to_a<64>(da, dp);
        float dq[16][4];
        zero_acc(dq);
        warp_gemm_rb<128, 64>(dq, da, sK, kLd, lane);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int row = r == 0 ? ra : rb;
          const int t = r == 0 ? ta : tb;
          if (t < 0) continue;
          float* dst = A.dq + (((size_t)b * d.S + t) * d.Hq + g * G + row % G) * kD + 2 * (lane % 4);
#pragma unroll
          for (int jt = 0; jt < 16; ++jt)
            add2(dst + 8 * jt, dq[jt][2 * r] * d.scale, dq[jt][2 * r + 1] * d.scale);
        }
      }
      __syncthreads();

      // ---- dV += P^T dO, dK += dS^T Q  (scale applied at the end)
      warp_gemm_atb<64, 128>(dv, sP, kLdh, km0, sdO + dn0, kLd, lane);
      warp_gemm_atb<64, 128>(dk, sdS, kLdh, km0, sQ + dn0, kLd, lane);

      // ---- student probabilities and dz (proxy rows x 64 keys, in 16 x 16 units)
      for (int u = warp; u < (TP / 16) * 4; u += 8) {
        const int mt = u / 4, nt = u % 4;
        float z[2][4];
        zero_acc(z);
        warp_gemm_abt<16, 128>(z, sQp + mt * 16 * kLd, kLd, sKp + nt * 16 * kLd, kLd, lane);
        const int pa_ = mt * 16 + lane / 4, pb_ = pa_ + 8;
        const int tpa = sTok[pa_], tpb = sTok[pb_];
#pragma unroll
        for (int jt = 0; jt < 2; ++jt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = e < 2 ? pa_ : pb_;
            const int t = e < 2 ? tpa : tpb;
            const int col = nt * 16 + 8 * jt + 2 * (lane % 4) + (e & 1);
            const int j = j0 + col;
            float dz = 0.f;
            if (t >= 0 && j <= t) {
              const float ppx = exp2f(z[jt][e] * sl2 - sLpx[row]);
              dz = A.cz * (ppx - sPbar[row * 64 + col]);
            }
            z[jt][e] = dz;
          }
#pragma unroll
        for (int jt = 0; jt < 2; ++jt) {
          const int col = nt * 16 + 8 * jt + 2 * (lane % 4);
          *reinterpret_cast<uint32_t*>(sdz + pa_ * kLdh + col) = pack_bf16(z[jt][0], z[jt][1]);
          *reinterpret_cast<uint32_t*>(sdz + pb_ * kLdh + col) = pack_bf16(z[jt][2], z[jt][3]);
        }
      }
      __syncthreads();

      // ---- dQp = scale dz Kp (fp32 atomics), dKp += dz^T Qp
      for (int u = warp; u < (TP / 16) * 2; u += 8) {
        const int mt = u / 2, nh = u % 2;
        float acc[8][4];
        zero_acc(acc);
        warp_gemm_ab<64, 64>(acc, sdz + mt * 16 * kLdh, kLdh, sKp + nh * 64, kLd, lane);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int row = mt * 16 + lane / 4 + 8 * r;
          const int t = sTok[row];
          if (t < 0) continue;
          float* dst = A.dqp + (((size_t)b * d.S + t) * d.Hp + g) * kD + nh * 64 + 2 * (lane % 4);
#pragma unroll
          for (int jt = 0; jt < 8; ++jt)
            add2(dst + 8 * jt, acc[jt][2 * r] * d.scale, acc[jt][2 * r + 1] * d.scale);
        }
      }
      warp_gemm_atb<64, TP>(dkp, sdz, kLdh, km0, sQp + dn0, kLd, lane);
      __syncthreads();
    }

    // ---- item epilogue: dK (scaled), dV, dKp (scaled) into the fp32 accumulators
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int j = j0 + km0 + lane / 4 + 8 * r;
      float* pk = A.dk + (((size_t)b * d.S + j) * d.Hkv + g) * kD + dn0 + 2 * (lane % 4);
      float* pv = A.dv + (((size_t)b * d.S + j) * d.Hkv + g) * kD + dn0 + 2 * (lane % 4);
      float* pkp = A.dkp + ((size_t)b * d.S + j) * kD + dn0 + 2 * (lane % 4);
#pragma unroll
      for (int jt = 0; jt < 8; ++jt) {
        add2(pk + 8 * jt, dk[jt][2 * r] * d.scale, dk[jt][2 * r + 1] * d.scale);
        add2(pv + 8 * jt, dv[jt][2 * r], dv[jt][2 * r + 1]);
        add2(pkp + 8 * jt, dkp[jt][2 * r] * d.scale, dkp[jt][2 * r + 1] * d.scale);
      }
    }
    __syncthreads();
  }
}

template <int G, bool kDense>
static void fused_bwd_g(const BwdArgs& a, cudaStream_t st) {
  constexpr int TT = 128 / G;
  constexpr int TP = TT < 16 ? 16 : TT;
  const size_t smem = (size_t)(3 * 64 + 2 * 128 + TP) * kLd * sizeof(bf16) +
                      (size_t)(2 * 128 + TP) * kLdh * sizeof(bf16) +
                      (size_t)(TP * 64 + 2 * 128 + TP) * sizeof(float) + TP * sizeof(int);
  cudaFuncSetAttribute(fused_bwd_kernel<G, kDense>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smem);
  fused_bwd_kernel<G, kDense><<<num_sms(), 256, smem, st>>>(a);
}

void launch_bwd_rowdot(const Dims& d, const void* o, const void* dout, float* drow,
                       cudaStream_t st) {
  const long long rows = (long long)d.B * d.S * d.Hq;
  long long grid = (rows * 32 + 255) / 256;
  if (grid > (long long)num_sms() * 16) grid = (long long)num_sms() * 16;
  rowdot_kernel<<<(int)grid, 256, 0, st>>>(d, (const bf16*)o, (const bf16*)dout, drow);
}

void launch_fused_bwd(const Dims& d, bool dense, const void* q, const void* k, const void* v,
                      const void* qp, const void* kp, const void* dout, const float* lse,
                      const float* drow, const float* lse_px, float kl_grad,
                      const int* seg_offset, const int* entries, const Item* items,
                      const int* n_items, long long max_items, float* dq_acc, float* dk_acc,
                      float* dv_acc, float* dqp_acc, float* dkp_acc, cudaStream_t st) {
  BwdArgs a;
  a.d = d;
  a.q = (const bf16*)q;
  a.k = (const bf16*)k;
  a.v = (const bf16*)v;
  a.qp = (const bf16*)qp;
  a.kp = (const bf16*)kp;
  a.dout = (const bf16*)dout;
  a.lse = lse;
  a.drow = drow;
  a.lse_px = lse_px;
  a.cz = (float)((double)kl_grad / ((double)d.B * d.S * d.Hp));
  a.seg_offset = seg_offset;
  a.entries = entries;
  a.items = items;
  a.n_items = n_items;
  a.max_items = max_items;
  a.dq = dq_acc;
  a.dk = dk_acc;
  a.dv = dv_acc;
  a.dqp = dqp_acc;
  a.dkp = dkp_acc;
#define MSA_BWD_CASE(GG)                           \
  case GG:                                         \
    if (dense)                                     \
      fused_bwd_g<GG, true>(a, st);                \
    else                                           \
      fused_bwd_g<GG, false>(a, st);               \
    break;
  switch (d.G) {
    MSA_BWD_CASE(2)
    MSA_BWD_CASE(4)
    MSA_BWD_CASE(8)
    MSA_BWD_CASE(16)
  }
#undef MSA_BWD_CASE
}

}  // namespace msa
