// Forward kernels on CUDA cores and warp-level m16n8k16 tensor-core products:
//   combine_kernel            second phase of the sparse forward (attn_fwd.cu writes the
//                             per-(token, head, slot) partials it merges)
//   dense_fwd_kernel          dense causal forward of the warmup mode
//   proxy_lse_*_kernel        proxy normaliser used by the backward (sparse over the selected
//                             blocks, dense over the causal prefix)
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace msa {

__device__ __forceinline__ float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x + __shfl_xor_sync(0xffffffffu, x, 2);
}

// Same validity rule as the index kernels: blocks ascending, within 0..t/128, -1 padding last.
__device__ __forceinline__ bool slot_valid(const int32_t* row, int s, int t, int& prev, bool& padded) {
  const int n = row[s];
  if (n < 0) {
    padded = true;
    return false;
  }
  if (padded || n <= prev || n > t / kBlock) return false;
  prev = n;
  return true;
}

// One 64-key step of online softmax for the warp's 16 rows.
//   s: raw scores (16 x 64); rows' token positions ta/tb decide the causal mask at key j0 + col.
template <bool kMask>
__device__ __forceinline__ void online_step(float (&s)[8][4], float (&m)[2], float (&l)[2],
                                            float (&o)[16][4], const bf16* sv, int ldv, int j0,
                                            int ta, int tb, float sl2, int lane) {
  float mx[2] = {m[0], m[1]};
#pragma unroll
  for (int jt = 0; jt < 8; ++jt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = j0 + 8 * jt + 2 * (lane % 4) + (e & 1);
      float x = s[jt][e] * sl2;
      if (kMask && j > (e < 2 ? ta : tb)) x = -INFINITY;
      s[jt][e] = x;
      mx[e >> 1] = fmaxf(mx[e >> 1], x);
    }
  }
  mx[0] = quad_max(mx[0]);
  mx[1] = quad_max(mx[1]);
  float alpha[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    alpha[r] = (m[r] == -INFINITY) ? 0.f : exp2f(m[r] - mx[r]);
    m[r] = mx[r];
    l[r] *= alpha[r];
  }
#pragma unroll
  for (int jt = 0; jt < 16; ++jt) {
    o[jt][0] *= alpha[0];
    o[jt][1] *= alpha[0];
    o[jt][2] *= alpha[1];
    o[jt][3] *= alpha[1];
  }
#pragma unroll
  for (int jt = 0; jt < 8; ++jt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float mm = m[e >> 1];
      const float p = (mm == -INFINITY) ? 0.f : exp2f(s[jt][e] - mm);
      s[jt][e] = p;
      l[e >> 1] += p;
    }
  }
  uint32_t pa[4][4];
  c_to_a<64>(pa, s);
  warp_gemm_rb<128, 64>(o, pa, sv, ldv, lane);
}

// ------------------------------------------------------------------------------------------
// Combine (second phase of the sparse forward): one warp per (b, t, h) merges the partials of
// its valid slots,  O = sum_s w_s O_s / sum_s w_s,  w_s = exp(lse_s - max),  LSE = max + log sum.
// A slot is valid iff its partial log-sum-exp was written: the workspace holds NaN (all-ones
// bytes) elsewhere.  Half-warps take alternate slots with 16-byte loads (8 columns per lane).
__global__ void __launch_bounds__(256, 3) combine_kernel(Dims d, const bf16* __restrict__ opart,
                                                      const float* __restrict__ lpart,
                                                      bf16* __restrict__ o, float* __restrict__ lse) {
  const long long rows = (long long)d.B * d.S * d.Hq;
  const int lane = threadIdx.x % 32, half = lane >> 4, l16 = lane & 15;
  const uint64_t pol = l2_policy_evict_first();  // each partial is read exactly once
  for (long long r = (blockIdx.x * (long long)blockDim.x + threadIdx.x) / 32; r < rows;
       r += (long long)gridDim.x * blockDim.x / 32) {
    const size_t base = (size_t)r * d.top_k;
    float l0 = lane < d.top_k ? lpart[base + lane] : NAN;
    float l1 = lane + 32 < d.top_k ? lpart[base + lane + 32] : NAN;
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
    // 16 slots per pass: all eight 16-byte loads of a lane are issued before any is used, and
    // they do not wait for the weights (a slot that was never written is loaded but not used)
    for (int s0 = 0; s0 < d.top_k; s0 += 16) {
      uint4 pv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int s = s0 + 2 * u + half;
        pv[u] = s < d.top_k ? ld_global_nc_v4_hint(opart + (base + s) * kD + l16 * 8, pol)
                            : make_uint4(0u, 0u, 0u, 0u);
      }
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
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 16);
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    if (half == 0)
      *reinterpret_cast<uint4*>(o + (size_t)r * kD + l16 * 8) =
          make_uint4(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv),
                     pack_bf16(acc[4] * inv, acc[5] * inv), pack_bf16(acc[6] * inv, acc[7] * inv));
    if (lane == 0) {
      const int h = (int)(r % d.Hq);
      const long long bt = r / d.Hq;
      const int t = (int)(bt % d.S), b = (int)(bt / d.S);
      lse[((size_t)b * d.Hq + h) * d.S + t] = sum > 0.f ? mx + logf(sum) : -INFINITY;
    }
  }
}

// ------------------------------------------------------------------------------------------
// Dense causal forward (warmup): a tile is 128/G consecutive tokens x the G heads of group g;
// keys stream in 64-key chunks, double-buffered.
template <int G>
__global__ void __launch_bounds__(256, 2)
    dense_fwd_kernel(Dims d, const bf16* __restrict__ q, const bf16* __restrict__ k,
                     const bf16* __restrict__ v, bf16* __restrict__ o, float* __restrict__ lse) {
  constexpr int TT = 128 / G;
  extern __shared__ __align__(128) uint8_t smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  bf16* sK = sQ + 128 * kLd;      // [2][64][kLd]
  bf16* sV = sK + 2 * 64 * kLd;   // [2][64][kLd]
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int ntile = d.S / TT;
  const int bg = blockIdx.x % (d.B * d.Hkv);
  const int tile = ntile - 1 - blockIdx.x / (d.B * d.Hkv);  // longest rows first
  const int b = bg / d.Hkv, g = bg % d.Hkv;
  const int t0 = tile * TT;
  const float sl2 = d.scale * kLog2e;
  load_rows_async(sQ, 128, [&](int r) -> const bf16* {
    return q + (((size_t)b * d.S + t0 + r / G) * d.Hq + g * G + r % G) * kD;
  }, tid, 256, q);
  const int nchunk = (t0 + TT + 63) / 64;
  auto load_chunk = [&](int c, int buf) {
    load_rows_async(sK + buf * 64 * kLd, 64, [&](int r) -> const bf16* {
      return k + (((size_t)b * d.S + c * 64 + r) * d.Hkv + g) * kD;
    }, tid, 256, k);
    load_rows_async(sV + buf * 64 * kLd, 64, [&](int r) -> const bf16* {
      return v + (((size_t)b * d.S + c * 64 + r) * d.Hkv + g) * kD;
    }, tid, 256, v);
  };
  load_chunk(0, 0);
  cp_async_commit();
  const int ra = warp * 16 + lane / 4, rb = ra + 8;
  const int ta = t0 + ra / G, tb = t0 + rb / G;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float oacc[16][4];
  zero_acc(oacc);
#pragma unroll 1
  for (int c = 0; c < nchunk; ++c) {
    if (c + 1 < nchunk) {
      load_chunk(c + 1, (c + 1) & 1);
      cp_async_commit();
      cp_async_wait_group<1>();
    } else {
      cp_async_wait_group<0>();
    }
    __syncthreads();
    float s[8][4];
    zero_acc(s);
    warp_gemm_abt<64, 128>(s, sQ + warp * 16 * kLd, kLd, sK + (c & 1) * 64 * kLd, kLd, lane);
    if ((c + 1) * 64 - 1 > t0)  // chunk reaches past the first token of the tile: mask
      online_step<true>(s, m, l, oacc, sV + (c & 1) * 64 * kLd, kLd, c * 64, ta, tb, sl2, lane);
    else
      online_step<false>(s, m, l, oacc, sV + (c & 1) * 64 * kLd, kLd, c * 64, ta, tb, sl2, lane);
    __syncthreads();
  }
  l[0] = quad_sum(l[0]);
  l[1] = quad_sum(l[1]);
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = r == 0 ? ra : rb;
    const int t = t0 + row / G, h = g * G + row % G;
    const float inv = 1.f / l[r];
    bf16* dst = o + (((size_t)b * d.S + t) * d.Hq + h) * kD + 2 * (lane % 4);
#pragma unroll
    for (int jt = 0; jt < 16; ++jt)
      *reinterpret_cast<uint32_t*>(dst + 8 * jt) =
          pack_bf16(oacc[jt][2 * r] * inv, oacc[jt][2 * r + 1] * inv);
    if (lane % 4 == 0) lse[((size_t)b * d.Hq + h) * d.S + t] = (m[r] + log2f(l[r])) * kLn2;
  }
}

// ------------------------------------------------------------------------------------------
// Proxy normaliser, sparse: item = (b, g, block n) and <= 128 tokens (one proxy row each);
// writes the per-slot log-sum-exp of scale * qp . kp over the block's visible keys.
__global__ void __launch_bounds__(256, 2)
    proxy_lse_sparse_kernel(Dims d, const bf16* __restrict__ qp, const bf16* __restrict__ kp,
                            const int* __restrict__ seg_offset, const int* __restrict__ entries,
                            const Item* __restrict__ items, const int* __restrict__ n_items,
                            long long max_items, float* __restrict__ lpx_part) {
  extern __shared__ __align__(128) uint8_t smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  bf16* sK = sQ + 128 * kLd;
  int* sTok = reinterpret_cast<int*>(sK + 128 * kLd);
  int* sSlot = sTok + 128;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const float sl2 = d.scale * kLog2e;
  long long total = *n_items;
  if (total > max_items) total = max_items;
  for (long long it = blockIdx.x; it < total; it += gridDim.x) {
    const Item item = items[it];
    const int n = item.seg % d.nblk;
    const int bg = (int)((item.seg % d.nseg()) / d.nblk);
    const int b = bg / d.Hp, g = bg % d.Hp;
    if (tid < 128) {
      int t = -1, slot = 0;
      if (tid < item.count) {
        const int e = entries[seg_offset[item.seg] + item.first + tid];
        t = e >> 8;
        slot = e & 255;
      }
      sTok[tid] = t;
      sSlot[tid] = slot;
    }
    __syncthreads();
    load_rows_async(sQ, 128, [&](int r) -> const bf16* {
      const int t = sTok[r];
      return t < 0 ? nullptr : qp + (((size_t)b * d.S + t) * d.Hp + g) * kD;
    }, tid, 256, qp);
    load_rows_async(sK, 128, [&](int r) -> const bf16* {
      return kp + ((size_t)b * d.S + n * kBlock + r) * kD;
    }, tid, 256, kp);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    const int ra = warp * 16 + lane / 4, rb = ra + 8;
    int ta = sTok[ra], tb = sTok[rb];
    const bool va = ta >= 0, vb = tb >= 0;
    if (!va) ta = 0x7fffffff;
    if (!vb) tb = 0x7fffffff;
    float mx[2] = {-INFINITY, -INFINITY}, sm[2] = {0.f, 0.f};
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      float s[8][4];
      zero_acc(s);
      warp_gemm_abt<64, 128>(s, sQ + warp * 16 * kLd, kLd, sK + half * 64 * kLd, kLd, lane);
      float nm[2] = {mx[0], mx[1]};
#pragma unroll
      for (int jt = 0; jt < 8; ++jt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = n * kBlock + half * 64 + 8 * jt + 2 * (lane % 4) + (e & 1);
          float x = s[jt][e] * sl2;
          if (j > (e < 2 ? ta : tb)) x = -INFINITY;
          s[jt][e] = x;
          nm[e >> 1] = fmaxf(nm[e >> 1], x);
        }
      nm[0] = quad_max(nm[0]);
      nm[1] = quad_max(nm[1]);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        sm[r] *= (mx[r] == -INFINITY) ? 0.f : exp2f(mx[r] - nm[r]);
        mx[r] = nm[r];
      }
#pragma unroll
      for (int jt = 0; jt < 8; ++jt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sm[e >> 1] += (mx[e >> 1] == -INFINITY) ? 0.f : exp2f(s[jt][e] - mx[e >> 1]);
    }
    sm[0] = quad_sum(sm[0]);
    sm[1] = quad_sum(sm[1]);
    if (lane % 4 == 0) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (!(r == 0 ? va : vb)) continue;
        const int row = r == 0 ? ra : rb;
        const int t = sTok[row];
        lpx_part[(((size_t)b * d.Hp + g) * d.S + t) * d.top_k + sSlot[row]] =
            (mx[r] + log2f(sm[r])) * kLn2;
      }
    }
    __syncthreads();
  }
}

__global__ void proxy_lse_combine_kernel(Dims d, const int32_t* __restrict__ idx,
                                         const float* __restrict__ lpx_part, float* __restrict__ lse_px) {
  const long long rows = (long long)d.B * d.Hp * d.S;
  for (long long r = blockIdx.x * (long long)blockDim.x + threadIdx.x; r < rows;
       r += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(r % d.S);
    const int32_t* row = idx + r * d.top_k;
    const float* part = lpx_part + r * d.top_k;
    float mx = -INFINITY;
    int prev = -1;
    bool padded = false;
    for (int s = 0; s < d.top_k; ++s)
      if (slot_valid(row, s, t, prev, padded)) mx = fmaxf(mx, part[s]);
    float sum = 0.f;
    prev = -1;
    padded = false;
    if (mx != -INFINITY)
      for (int s = 0; s < d.top_k; ++s)
        if (slot_valid(row, s, t, prev, padded)) sum += expf(part[s] - mx);
    lse_px[r] = sum > 0.f ? mx + logf(sum) : -INFINITY;
  }
}

// Proxy normaliser, dense (warmup): 128 tokens of one group against every visible key.
__global__ void __launch_bounds__(256, 2)
    proxy_lse_dense_kernel(Dims d, const bf16* __restrict__ qp, const bf16* __restrict__ kp,
                           float* __restrict__ lse_px) {
  extern __shared__ __align__(128) uint8_t smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  bf16* sK = sQ + 128 * kLd;  // [2][64][kLd]
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int bg = blockIdx.x % (d.B * d.Hp);
  const int qb = d.nblk - 1 - blockIdx.x / (d.B * d.Hp);
  const int b = bg / d.Hp, g = bg % d.Hp;
  const int t0 = qb * kBlock;
  const float sl2 = d.scale * kLog2e;
  load_rows_async(sQ, 128, [&](int r) -> const bf16* {
    return qp + (((size_t)b * d.S + t0 + r) * d.Hp + g) * kD;
  }, tid, 256, qp);
  const int nchunk = (t0 + kBlock) / 64;
  auto load_chunk = [&](int c, int buf) {
    load_rows_async(sK + buf * 64 * kLd, 64, [&](int r) -> const bf16* {
      return kp + ((size_t)b * d.S + c * 64 + r) * kD;
    }, tid, 256, kp);
  };
  load_chunk(0, 0);
  cp_async_commit();
  const int ra = warp * 16 + lane / 4, rb = ra + 8;
  const int ta = t0 + ra, tb = t0 + rb;
  float mx[2] = {-INFINITY, -INFINITY}, sm[2] = {0.f, 0.f};
#pragma unroll 1
  for (int c = 0; c < nchunk; ++c) {
    if (c + 1 < nchunk) {
      load_chunk(c + 1, (c + 1) & 1);
      cp_async_commit();
      cp_async_wait_group<1>();
    } else {
      cp_async_wait_group<0>();
    }
    __syncthreads();
    float s[8][4];
    zero_acc(s);
    warp_gemm_abt<64, 128>(s, sQ + warp * 16 * kLd, kLd, sK + (c & 1) * 64 * kLd, kLd, lane);
    float nm[2] = {mx[0], mx[1]};
#pragma unroll
    for (int jt = 0; jt < 8; ++jt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = c * 64 + 8 * jt + 2 * (lane % 4) + (e & 1);
        float x = s[jt][e] * sl2;
        if (j > (e < 2 ? ta : tb)) x = -INFINITY;
        s[jt][e] = x;
        nm[e >> 1] = fmaxf(nm[e >> 1], x);
      }
    nm[0] = quad_max(nm[0]);
    nm[1] = quad_max(nm[1]);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      sm[r] *= (mx[r] == -INFINITY) ? 0.f : exp2f(mx[r] - nm[r]);
      mx[r] = nm[r];
    }
#pragma unroll
    for (int jt = 0; jt < 8; ++jt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        sm[e >> 1] += (mx[e >> 1] == -INFINITY) ? 0.f : exp2f(s[jt][e] - mx[e >> 1]);
    __syncthreads();
  }
  sm[0] = quad_sum(sm[0]);
  sm[1] = quad_sum(sm[1]);
  if (lane % 4 == 0) {
    lse_px[((size_t)b * d.Hp + g) * d.S + ta] = (mx[0] + log2f(sm[0])) * kLn2;
    lse_px[((size_t)b * d.Hp + g) * d.S + tb] = (mx[1] + log2f(sm[1])) * kLn2;
  }
}

// ------------------------------------------------------------------------------------------
static int persistent_grid(int ctas_per_sm) { return num_sms() * ctas_per_sm; }

void launch_combine(const Dims& d, const void* opart, const float* lpart, void* o, float* lse,
                    cudaStream_t st) {
  const long long rows = (long long)d.B * d.S * d.Hq;
  long long grid = (rows * 32 + 255) / 256;
  if (grid > (long long)num_sms() * 8) grid = (long long)num_sms() * 8;
  combine_kernel<<<(int)grid, 256, 0, st>>>(d, (const bf16*)opart, lpart, (bf16*)o, lse);
}

template <int G>
static void dense_fwd_g(const Dims& d, const void* q, const void* k, const void* v, void* o,
                        float* lse, cudaStream_t st) {
  const size_t smem = (128 + 4 * 64) * kLd * sizeof(bf16);
  cudaFuncSetAttribute(dense_fwd_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const int grid = (d.S / (128 / G)) * d.B * d.Hkv;
  dense_fwd_kernel<G><<<grid, 256, smem, st>>>(d, (const bf16*)q, (const bf16*)k, (const bf16*)v,
                                                (bf16*)o, lse);
}

void launch_dense_fwd(const Dims& d, const void* q, const void* k, const void* v, void* o,
                      float* lse, cudaStream_t st) {
  switch (d.G) {
    case 1: dense_fwd_g<1>(d, q, k, v, o, lse, st); break;
    case 2: dense_fwd_g<2>(d, q, k, v, o, lse, st); break;
    case 4: dense_fwd_g<4>(d, q, k, v, o, lse, st); break;
    case 8: dense_fwd_g<8>(d, q, k, v, o, lse, st); break;
    case 16: dense_fwd_g<16>(d, q, k, v, o, lse, st); break;
  }
}

void launch_proxy_lse_sparse(const Dims& d, const void* qp, const void* kp, const int* seg_offset,
                             const int* entries, const Item* items, const int* n_items,
                             long long max_items, float* lpx_part, cudaStream_t st) {
  const size_t smem = 2 * 128 * kLd * sizeof(bf16) + 2 * 128 * sizeof(int);
  cudaFuncSetAttribute(proxy_lse_sparse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  proxy_lse_sparse_kernel<<<persistent_grid(2), 256, smem, st>>>(
      d, (const bf16*)qp, (const bf16*)kp, seg_offset, entries, items, n_items, max_items, lpx_part);
}

void launch_proxy_lse_combine(const Dims& d, const int32_t* idx, const float* lpx_part,
                              float* lse_px, cudaStream_t st) {
  const long long rows = (long long)d.B * d.Hp * d.S;
  long long grid = (rows + 255) / 256;
  if (grid > (long long)num_sms() * 16) grid = (long long)num_sms() * 16;
  proxy_lse_combine_kernel<<<(int)grid, 256, 0, st>>>(d, idx, lpx_part, lse_px);
}

void launch_proxy_lse_dense(const Dims& d, const void* qp, const void* kp, float* lse_px,
                            cudaStream_t st) {
  const size_t smem = (128 + 2 * 64) * kLd * sizeof(bf16);
  cudaFuncSetAttribute(proxy_lse_dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  proxy_lse_dense_kernel<<<d.nblk * d.B * d.Hp, 256, smem, st>>>(d, (const bf16*)qp,
                                                                 (const bf16*)kp, lse_px);
}

}  // namespace msa
