// CUDA-core kernels of the forward and of the proxy normaliser:
//   combine_kernel            second phase of the sparse forward (attn_fwd.cu writes the
//                             per-(token, head, slot) partials it merges)
//   proxy_lse_combine_kernel  proxy normaliser of the backward from its per-slot partials (the
//                             tcgen05 sparse forward in proxy mode, attn_fwd.cu, writes them;
//                             the dense normaliser of the warmup backward is an epilogue of the
//                             selection kernel, topk.cu)
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {

// ------------------------------------------------------------------------------------------
// Combine (second phase of the sparse forward): one warp per (b, t, h) merges the partials of
// its valid slots,  O = sum_s w_s O_s / sum_s w_s,  w_s = exp(lse_s - max),  LSE = max + log sum.
// A slot is valid iff its partial log-sum-exp was written: the workspace holds NaN (all-ones
// bytes) elsewhere.  Half-warps take alternate slots with 16-byte loads (8 columns per lane).
// One pass covers the tokens [t0, t0 + tn) of every sequence, its partials indexed
// ((b tp + t - t0) Hq + h) top_k + slot.
__global__ void __launch_bounds__(256, 3) combine_kernel(Dims d, const bf16* __restrict__ opart,
                                                      const float* __restrict__ lpart,
                                                      bf16* __restrict__ o, float* __restrict__ lse,
                                                      int t0, int tn, int tp) {
  const long long rows = (long long)d.B * tn * d.Hq;
  const int lane = threadIdx.x % 32, half = lane >> 4, l16 = lane & 15;
  const uint64_t pol = l2_policy_evict_first();  // each partial is read exactly once
  for (long long r = (blockIdx.x * (long long)blockDim.x + threadIdx.x) / 32; r < rows;
       r += (long long)gridDim.x * blockDim.x / 32) {
    const int h = (int)(r % d.Hq);
    const long long bt = r / d.Hq;
    const int tr = (int)(bt % tn), b = (int)(bt / tn);  // token t0 + tr of sequence b
    const size_t base = (((size_t)b * tp + tr) * d.Hq + h) * d.top_k;
    const size_t orow = ((size_t)b * d.S + t0 + tr) * d.Hq + h;
    float l0 = lane < d.top_k ? lpart[base + lane] : NAN;
    float l1 = lane + 32 < d.top_k ? lpart[base + lane + 32] : NAN;
    // the first 16 slots' partials are requested together with the log-sum-exps, before the
    // weights are known (one memory round trip per row, not two)
    uint4 pv0[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int s = 2 * u + half;
      pv0[u] = s < d.top_k ? ld_global_nc_v4_hint(opart + (base + s) * kD + l16 * 8, pol)
                           : make_uint4(0u, 0u, 0u, 0u);
    }
    l0 = l0 == l0 ? l0 : -INFINITY;  // NaN: slot not written (invalid or padding)
    l1 = l1 == l1 ? l1 : -INFINITY;
    float mx = fmaxf(l0, l1);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float w0 = l0 == -INFINITY ? 0.f : expf(l0 - mx);
    const float w1 = l1 == -INFINITY ? 0.f : expf(l1 - mx);
    float sum = w0 + w1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    auto accumulate = [&](int s0, const uint4 (&pv)[8]) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int s = s0 + 2 * u + half;
        const float a = __shfl_sync(0xffffffffu, w0, s & 31);
        const float c = __shfl_sync(0xffffffffu, w1, s & 31);
        const float w = s < 32 ? a : c;
        if (s < d.top_k && w > 0.f) {
          const uint32_t pw[4] = {pv[u].x, pv[u].y, pv[u].z, pv[u].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162*>(&pw[e]);
            acc[2 * e] += w * __low2float(p2);
            acc[2 * e + 1] += w * __high2float(p2);
          }
        }
      }
    };
    accumulate(0, pv0);
    // further passes of 16 slots (top_k > 16): all eight 16-byte loads of a lane are issued
    // before any is used (a slot that was never written is loaded but not used)
    for (int s0 = 16; s0 < d.top_k; s0 += 16) {
      uint4 pv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int s = s0 + 2 * u + half;
        pv[u] = s < d.top_k ? ld_global_nc_v4_hint(opart + (base + s) * kD + l16 * 8, pol)
                            : make_uint4(0u, 0u, 0u, 0u);
      }
      accumulate(s0, pv);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 16);
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    if (half == 0)
      *reinterpret_cast<uint4*>(o + orow * kD + l16 * 8) =
          make_uint4(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv),
                     pack_bf16(acc[4] * inv, acc[5] * inv), pack_bf16(acc[6] * inv, acc[7] * inv));
    if (lane == 0) lse[((size_t)b * d.Hq + h) * d.S + t0 + tr] = sum > 0.f ? mx + logf(sum) : -INFINITY;
  }
}

// Proxy normaliser from its per-slot partials (attn_fwd.cu, proxy mode): lpx_part[(b S + t) Hp + g]
// [slot] holds the log-sum-exp over that slot's visible keys, or NaN (all-ones bytes) where no list
// entry wrote it (padding); LSE_px[(b Hp + g) S + t] = log sum_slot exp(partial).
__global__ void proxy_lse_combine_kernel(Dims d, const float* __restrict__ lpx_part,
                                         float* __restrict__ lse_px) {
  const long long rows = (long long)d.B * d.S * d.Hp;
  for (long long r = blockIdx.x * (long long)blockDim.x + threadIdx.x; r < rows;
       r += (long long)gridDim.x * blockDim.x) {
    const float* part = lpx_part + r * d.top_k;
    float mx = -INFINITY;
    for (int s = 0; s < d.top_k; ++s) {
      const float v = part[s];
      if (v == v) mx = fmaxf(mx, v);
    }
    float sum = 0.f;
    if (mx != -INFINITY)
      for (int s = 0; s < d.top_k; ++s) {
        const float v = part[s];
        if (v == v) sum += expf(v - mx);
      }
    const int g = (int)(r % d.Hp);
    const long long bt = r / d.Hp;
    const int t = (int)(bt % d.S), b = (int)(bt / d.S);
    lse_px[((long long)b * d.Hp + g) * d.S + t] = sum > 0.f ? mx + logf(sum) : -INFINITY;
  }
}

// ------------------------------------------------------------------------------------------

void launch_combine(const Dims& d, const void* opart, const float* lpart, void* o, float* lse,
                    int t0, int tn, int tp, cudaStream_t st) {
  const long long rows = (long long)d.B * tn * d.Hq;
  long long grid = (rows * 32 + 255) / 256;
  if (grid > (long long)num_sms() * 8) grid = (long long)num_sms() * 8;
  combine_kernel<<<(int)grid, 256, 0, st>>>(d, (const bf16*)opart, lpart, (bf16*)o, lse, t0, tn, tp);
}



void launch_proxy_lse_combine(const Dims& d, const float* lpx_part, float* lse_px,
                              cudaStream_t st) {
  const long long rows = (long long)d.B * d.Hp * d.S;
  long long grid = (rows + 255) / 256;
  if (grid > (long long)num_sms() * 16) grid = (long long)num_sms() * 16;
  proxy_lse_combine_kernel<<<(int)grid, 256, 0, st>>>(d, lpx_part, lse_px);
}


}  // namespace msa
