// Proxy scores + causal block max-pool + streaming top-k (blog, "Forward > Proxy attention";
// forum summary, "Architecture" and "Exp-free TopK").
//
// A CTA owns the 128 tokens of query block qb for one group g.  Every key block n < qb is fully
// visible to all of them (the local block qb is forced in and never scored), so the causal mask
// reduces to "stream blocks 0 .. qb-1".  For each streamed block the tensor core forms the
// 128 x 128 raw score tile qp . kp in tensor memory (the positive scale does not change the
// order, so it is not applied); the epilogue max-pools each row over the block and inserts the
// block score into that row's running list of the best top_k - 1 non-local blocks, kept sorted
// in registers.  Ties keep the lower block: a new score enters only if strictly larger than the
// current last entry and is placed after equal entries.  No exponential is ever taken.
//
// Roles (256 threads): warp 0 issues the TMA loads (the query tile once, then a 4-deep ring of
// 128-key proxy-key blocks), warp 1 issues the MMAs (one thread), warp 2 owns the tensor memory
// (4 accumulators x 128 columns), warps 4..7 are the epilogue (thread i of warpgroup 1 owns
// score row i = TMEM lane i).
//
// The same pipeline with kLse = true is the dense proxy normaliser of the warmup backward (blog,
// "Warmup kernels": the indexer's log-sum-exp over the full causal prefix): blocks 0 .. qb, the
// local block included with its causal cut (key j visible to token t iff j <= t), and an epilogue
// that keeps per row a running maximum and sum of exponentials of scale * qp . kp and writes
// LSE_px[b, g, t] = log sum_{j <= t} exp(scale * qp_t . kp_j).
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tmap.h"

namespace msa {

namespace {
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr int kStages = 4;
constexpr int kAcc = 4;
constexpr int kTileBytes = 128 * 128 * 2;  // one 128 x 128 bf16 tile (two SW128 panels)

struct TopkSmem {
  uint64_t q_full;
  uint64_t kp_full[kStages], kp_empty[kStages];
  uint64_t acc_full[kAcc], acc_empty[kAcc];
  uint32_t tmem;
};
}  // namespace

// NH proxy heads per block (1 or 2): with two, each streamed proxy-key block feeds both heads'
// products and two epilogue warpgroups (warps 4-7 head 0, 8-11 head 1) share the SM sub-partitions.
template <int KMAX, bool kLse, int NH>
__global__ void __launch_bounds__(128 + 128 * NH, 1)
    proxy_topk_kernel(const __grid_constant__ CUtensorMap tm_qp,
                      const __grid_constant__ CUtensorMap tm_kp, Dims d,
                      int32_t* __restrict__ idx, float* __restrict__ lse_out,
                      unsigned* __restrict__ status) {
  using namespace sm100;
  constexpr int kAccH = kAcc / NH;  // accumulators per head
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* sQ = base;                      // NH x 32 KB
  uint8_t* sK = base + NH * kTileBytes;    // kStages x 32 KB
  TopkSmem* sh = reinterpret_cast<TopkSmem*>(sK + kStages * kTileBytes);

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int hpb = d.Hp / NH;  // head pairs (or heads) per batch row
  const int nbg = d.B * hpb;
  const int qb = d.nblk - 1 - blockIdx.x / nbg;  // most work first
  const int bg = blockIdx.x % nbg;
  const int b = bg / hpb, g0 = (bg % hpb) * NH;
  const int t0 = qb * kBlock;
  const int KL = d.top_k - 1;
  const int nb = kLse ? qb + 1 : qb;  // key blocks streamed

  if (tid == 0) {
    mbar_init(&sh->q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh->kp_full[i], 1);
      mbar_init(&sh->kp_empty[i], 1);
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(&sh->acc_full[i], 1);
      mbar_init(&sh->acc_empty[i], 4);
    }
    mbar_fence_init();
  }
  if (warp == 2) {
    tmem_alloc(&sh->tmem, 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = sh->tmem;
  const uint32_t sQa = static_cast<uint32_t>(__cvta_generic_to_shared(sQ));
  const uint32_t sKa = static_cast<uint32_t>(__cvta_generic_to_shared(sK));

  if (warp == 0 && lane == 0 && nb > 0) {
    // ---- producer
    tma_prefetch_desc(&tm_qp);
    tma_prefetch_desc(&tm_kp);
    mbar_expect_tx(&sh->q_full, NH * kTileBytes);
    for (int h = 0; h < NH; ++h) {
      tma_load_3d(sQ + h * kTileBytes, &tm_qp, 0, g0 + h, b * d.S + t0, &sh->q_full);
      tma_load_3d(sQ + h * kTileBytes + kTileBytes / 2, &tm_qp, 64, g0 + h, b * d.S + t0, &sh->q_full);
    }
    for (int n = 0; n < nb; ++n) {
      const int s = n % kStages;
      if (n >= kStages && !mbar_wait(&sh->kp_empty[s], ((n / kStages) - 1) & 1, status)) break;
      uint8_t* dst = sK + s * kTileBytes;
      mbar_expect_tx(&sh->kp_full[s], kTileBytes);
      tma_load_2d(dst, &tm_kp, 0, b * d.S + n * kBlock, &sh->kp_full[s]);
      tma_load_2d(dst + kTileBytes / 2, &tm_kp, 64, b * d.S + n * kBlock, &sh->kp_full[s]);
    }
  } else if (warp == 1 && lane == 0 && nb > 0) {
    // ---- MMA issuer
    constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
    bool ok = mbar_wait(&sh->q_full, 0, status);
    for (int n = 0; ok && n < nb; ++n) {
      const int s = n % kStages;
      if (!mbar_wait(&sh->kp_full[s], (n / kStages) & 1, status)) break;
      const uint32_t kaddr = sKa + s * kTileBytes;
      for (int h = 0; h < NH; ++h) {
        const int a = h * kAccH + n % kAccH;
        if (n >= kAccH && !mbar_wait(&sh->acc_empty[a], ((n / kAccH) - 1) & 1, status)) {
          ok = false;
          break;
        }
        fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ss(tmem + a * 128, desc_kmajor(sQa + h * kTileBytes, 128, ks),
                 desc_kmajor(kaddr, 128, ks), idesc, ks > 0);
        mma_commit(&sh->acc_full[a]);
      }
      if (!ok) break;
      mma_commit(&sh->kp_empty[s]);
    }
  } else if (warp >= 4 && kLse) {
    // ---- normaliser epilogue: thread owns score row `row` (token t0 + row) of head g0 + hh
    const int q4 = warp % 4, hh = (warp - 4) >> 2;
    const int row = q4 * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const float sl2 = d.scale * kLog2e;
    float m = -INFINITY, l = 0.f;  // running max of the raw scores, sum of exp2(sl2 (z - m))
    for (int n = 0; n < nb; ++n) {
      const int a = hh * kAccH + n % kAccH;
      const int lim = n == qb ? row : kBlock - 1;  // visible columns 0 .. lim
      __syncwarp();
      if (!mbar_wait_warp(&sh->acc_full[a], (n / kAccH) & 1, status)) break;
      fence_after_sync();
      float m8[8];  // independent running maxima (no long dependency chain)
#pragma unroll
      for (int u = 0; u < 8; ++u) m8[u] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; c += 2) {
        uint32_t r0[32], r1[32];
        tmem_ld32(tmem + lane_base + a * 128 + c * 32, r0);
        tmem_ld32(tmem + lane_base + a * 128 + (c + 1) * 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          m8[j & 7] = fmaxf(m8[j & 7], fmaxf(c * 32 + j <= lim ? __uint_as_float(r0[j]) : -INFINITY,
                                             (c + 1) * 32 + j <= lim ? __uint_as_float(r1[j]) : -INFINITY));
      }
      const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      if (mx > m) {  // column 0 is always visible, so mx is finite
        l *= ex2_approx((m - mx) * sl2);  // m = -inf: l = 0 anyway
        m = mx;
      }
      const float mb = m * sl2;
      float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 4; c += 2) {
        uint32_t r0[32], r1[32];
        tmem_ld32(tmem + lane_base + a * 128 + c * 32, r0);
        tmem_ld32(tmem + lane_base + a * 128 + (c + 1) * 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          // exponentiate unconditionally, then select: no per-lane branches
          const float e0 = ex2_approx(fmaf(__uint_as_float(r0[j]), sl2, -mb));
          const float e1 = ex2_approx(fmaf(__uint_as_float(r1[j]), sl2, -mb));
          s8[j & 7] += (c * 32 + j <= lim ? e0 : 0.f) + ((c + 1) * 32 + j <= lim ? e1 : 0.f);
        }
      }
      l += ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->acc_empty[a]);
    }
    lse_out[((size_t)b * d.Hp + g0 + hh) * d.S + t0 + row] = (m * sl2 + __log2f(l)) * kLn2;
  } else if (warp >= 4) {
    // ---- epilogue: thread owns score row `row` of head g0 + hh
    const int q4 = warp % 4, hh = (warp - 4) >> 2;
    const int row = q4 * 32 + lane;
    float vals[KMAX - 1];
    int ids[KMAX - 1];
#pragma unroll
    for (int p = 0; p < KMAX - 1; ++p) {
      vals[p] = -INFINITY;
      ids[p] = -1;
    }
    float kth = -INFINITY;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    for (int n = 0; n < qb; ++n) {
      const int a = hh * kAccH + n % kAccH;
      __syncwarp();
      if (!mbar_wait_warp(&sh->acc_full[a], (n / kAccH) & 1, status)) break;
      fence_after_sync();
      // eight independent running maxima: a single one would be a 128-step dependency chain
      float m8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) m8[u] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; c += 2) {
        uint32_t r0[32], r1[32];
        tmem_ld32(tmem + lane_base + a * 128 + c * 32, r0);
        tmem_ld32(tmem + lane_base + a * 128 + (c + 1) * 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          m8[j & 7] = fmaxf(m8[j & 7], fmaxf(__uint_as_float(r0[j]), __uint_as_float(r1[j])));
      }
      const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->acc_empty[a]);
      if (mx > kth) {
        // sorted insert (descending); after the insertion point every entry shifts down one
        float cv = mx;
        int ci = n;
        bool ins = false;
#pragma unroll
        for (int p = 0; p < KMAX - 1; ++p) {
          if (p < KL) {
            const bool take = ins || cv > vals[p];
            const float tv = vals[p];
            const int ti = ids[p];
            vals[p] = take ? cv : tv;
            ids[p] = take ? ci : ti;
            cv = take ? tv : cv;
            ci = take ? ti : ci;
            ins = take;
            if (p == KL - 1) kth = vals[p];
          }
        }
      }
    }
    // emit: picked non-local blocks ascending, then the local block, then -1 padding
    int sel[KMAX];
    int nv = 0;
#pragma unroll
    for (int p = 0; p < KMAX - 1; ++p)
      if (p < KL && ids[p] >= 0) sel[nv++] = ids[p];
    for (int i = 1; i < nv; ++i) {
      const int x = sel[i];
      int j = i - 1;
      while (j >= 0 && sel[j] > x) {
        sel[j + 1] = sel[j];
        --j;
      }
      sel[j + 1] = x;
    }
    int32_t* out = idx + (((size_t)b * d.Hp + g0 + hh) * d.S + t0 + row) * d.top_k;
    for (int i = 0; i < d.top_k; ++i) out[i] = i < nv ? sel[i] : (i == nv ? qb : -1);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 2) tmem_dealloc(tmem, 512);
}

template <int KMAX, bool kLse, int NH>
static void topk_launch_nh(const CUtensorMap& mq, const CUtensorMap& mk, const Dims& d, int32_t* idx,
                           float* lse, unsigned* status, cudaStream_t st) {
  const size_t smem = 1024 + (NH + kStages) * kTileBytes + sizeof(TopkSmem);
  cudaFuncSetAttribute(proxy_topk_kernel<KMAX, kLse, NH>,
                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  proxy_topk_kernel<KMAX, kLse, NH><<<d.B * (d.Hp / NH) * d.nblk, 128 + 128 * NH, smem, st>>>(
      mq, mk, d, idx, lse, status);
}
// Two proxy heads per block when the head count is even and the epilogue's registers allow it
// (lists of up to 15 blocks, or the normaliser); one otherwise.
template <int KMAX, bool kLse>
static void topk_launch(const CUtensorMap& mq, const CUtensorMap& mk, const Dims& d, int32_t* idx,
                        float* lse, unsigned* status, cudaStream_t st) {
  if constexpr (KMAX <= 16) {
    if (d.Hp % 2 == 0) {
      topk_launch_nh<KMAX, kLse, 2>(mq, mk, d, idx, lse, status, st);
      return;
    }
  }
  topk_launch_nh<KMAX, kLse, 1>(mq, mk, d, idx, lse, status, st);
}

static bool proxy_maps(const Dims& d, const void* qp, const void* kp, CUtensorMap* mq, CUtensorMap* mk) {
  const uint64_t qdims[3] = {128, (uint64_t)d.Hp, (uint64_t)d.B * d.S};
  const uint64_t qstr[2] = {128 * 2, (uint64_t)d.Hp * 128 * 2};
  const uint32_t qbox[3] = {64, 1, 128};
  const uint64_t kdims[2] = {128, (uint64_t)d.B * d.S};
  const uint64_t kstr[1] = {128 * 2};
  const uint32_t kbox[2] = {64, 128};
  return make_tmap_bf16(mq, qp, 3, qdims, qstr, qbox) && make_tmap_bf16(mk, kp, 2, kdims, kstr, kbox);
}

bool launch_proxy_topk(const Dims& d, const void* qp, const void* kp, int32_t* idx,
                       unsigned* status, cudaStream_t st) {
  CUtensorMap mq, mk;
  if (!proxy_maps(d, qp, kp, &mq, &mk)) return false;
  if (d.top_k <= 8)
    topk_launch<8, false>(mq, mk, d, idx, nullptr, status, st);
  else if (d.top_k <= 16)
    topk_launch<16, false>(mq, mk, d, idx, nullptr, status, st);
  else if (d.top_k <= 32)
    topk_launch<32, false>(mq, mk, d, idx, nullptr, status, st);
  else
    topk_launch<64, false>(mq, mk, d, idx, nullptr, status, st);
  return true;
}

bool launch_proxy_lse_dense(const Dims& d, const void* qp, const void* kp, float* lse_px,
                            unsigned* status, cudaStream_t st) {
  CUtensorMap mq, mk;
  if (!proxy_maps(d, qp, kp, &mq, &mk)) return false;
  topk_launch<2, true>(mq, mk, d, nullptr, lse_px, status, st);
  return true;
}

}  // namespace msa
