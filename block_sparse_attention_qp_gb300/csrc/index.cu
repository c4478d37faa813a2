// Index inversion and work-list construction (integer, HBM/latency bound).
//
// The blog ("Backward") inverts the cached map  (batch, proxy head, query, slot) -> key block
// into  (batch, proxy head, key block) -> queries that use the block, and schedules work per key
// block so that the block's keys and values are loaded once for many queries.  Here the inverse
// map is a CSR structure: one list per (chunk c, b, g, n) of packed entries (t << 8 | slot), where
// chunk c holds the tokens [c * chunk, (c+1) * chunk).  Lists are numbered chunk-major, so work
// items running at the same time touch the gradient rows of one chunk only (which then stay in
// L2).  Lists are cut into fixed-size items that the attention kernels consume.
#include "common.cuh"
#include "kernels.h"

namespace msa {

// Validity of entry s of a block_idx row: 0 <= n <= t/128, strictly ascending, and -1 only as
// trailing padding.  Returns the block or -1 (padding or invalid); *bad is set for invalid.
__device__ __forceinline__ int checked_block(const int32_t* row, int s, int t, int& prev,
                                             bool& padded, bool& bad) {
  const int n = row[s];
  if (n < 0) {
    if (n != -1) bad = true;
    padded = true;
    return -1;
  }
  if (padded || n <= prev || n > t / kBlock) {
    bad = true;
    return -1;
  }
  prev = n;
  return n;
}

__global__ void count_kernel(Dims d, const int32_t* __restrict__ idx, int* __restrict__ seg_count,
                             unsigned* status) {
  const long long rows = (long long)d.B * d.Hp * d.S;
  for (long long r = blockIdx.x * (long long)blockDim.x + threadIdx.x; r < rows;
       r += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(r % d.S);
    const long long bg = r / d.S;  // b * Hp + g
    const int32_t* row = idx + r * d.top_k;
    int prev = -1;
    bool padded = false, bad = false;
    for (int s = 0; s < d.top_k; ++s) {
      const int n = checked_block(row, s, t, prev, padded, bad);
      if (n >= 0) atomicAdd(seg_count + (long long)(t / d.chunk) * d.nseg() + bg * d.nblk + n, 1);
    }
    if (bad) atomicOr(status, kStatusBadIndex);
  }
}

__global__ void fill_kernel(Dims d, const int32_t* __restrict__ idx, const int* __restrict__ seg_offset,
                            int* __restrict__ seg_cursor, int* __restrict__ entries) {
  const long long rows = (long long)d.B * d.Hp * d.S;
  for (long long r = blockIdx.x * (long long)blockDim.x + threadIdx.x; r < rows;
       r += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(r % d.S);
    const long long bg = r / d.S;
    const int32_t* row = idx + r * d.top_k;
    int prev = -1;
    bool padded = false, bad = false;
    for (int s = 0; s < d.top_k; ++s) {
      const int n = checked_block(row, s, t, prev, padded, bad);
      if (n < 0) continue;
      const long long seg = (long long)(t / d.chunk) * d.nseg() + bg * d.nblk + n;
      const int pos = atomicAdd(seg_cursor + seg, 1);
      entries[seg_offset[seg] + pos] = (t << 8) | s;
    }
  }
}

// The same two steps with the counting done in shared memory first, for key-block counts up to
// kHistBlocks: a block takes the 128 rows of one (b, g) and one sequence chunk (S and the chunk
// are multiples of 128), so all its entries fall in the lists of one (c, b, g), and many tokens
// share a block (their local block, blocks most of them select).  The block adds each non-zero
// count to the global list once -- one global atomic per (block, key block) instead of one per
// entry -- and, when filling, reserves each list's range once and places its entries from
// shared cursors.
constexpr int kHistRows = 128, kHistBlocks = 2048;

__global__ void __launch_bounds__(kHistRows) count_hist_kernel(Dims d, const int32_t* __restrict__ idx,
                                                               int* __restrict__ seg_count, unsigned* status) {
  __shared__ int hist[kHistBlocks];
  const long long r = (long long)blockIdx.x * kHistRows + threadIdx.x;
  const long long r0 = (long long)blockIdx.x * kHistRows;
  const int t0 = (int)(r0 % d.S), t = (int)(r % d.S);
  const long long bg = r0 / d.S;
  const int nmax = min(d.nblk, (t0 + kHistRows - 1) / kBlock + 1);  // blocks these tokens may use
  for (int i = threadIdx.x; i < nmax; i += kHistRows) hist[i] = 0;
  __syncthreads();
  const int32_t* row = idx + r * d.top_k;
  int prev = -1;
  bool padded = false, bad = false;
  for (int s = 0; s < d.top_k; ++s) {
    const int n = checked_block(row, s, t, prev, padded, bad);
    if (n >= 0) atomicAdd(&hist[n], 1);
  }
  if (bad) atomicOr(status, kStatusBadIndex);
  __syncthreads();
  int* dst = seg_count + (long long)(t0 / d.chunk) * d.nseg() + bg * d.nblk;
  for (int i = threadIdx.x; i < nmax; i += kHistRows)
    if (hist[i]) atomicAdd(dst + i, hist[i]);
}

__global__ void __launch_bounds__(kHistRows) fill_hist_kernel(Dims d, const int32_t* __restrict__ idx,
                                                              const int* __restrict__ seg_offset,
                                                              int* __restrict__ seg_cursor, int* __restrict__ entries) {
  __shared__ int base[kHistBlocks], cur[kHistBlocks];
  const long long r = (long long)blockIdx.x * kHistRows + threadIdx.x;
  const long long r0 = (long long)blockIdx.x * kHistRows;
  const int t0 = (int)(r0 % d.S), t = (int)(r % d.S);
  const long long bg = r0 / d.S;
  const int nmax = min(d.nblk, (t0 + kHistRows - 1) / kBlock + 1);
  for (int i = threadIdx.x; i < nmax; i += kHistRows) {
    base[i] = 0;
    cur[i] = 0;
  }
  __syncthreads();
  const int32_t* row = idx + r * d.top_k;
  {
    int prev = -1;
    bool padded = false, bad = false;
    for (int s = 0; s < d.top_k; ++s) {
      const int n = checked_block(row, s, t, prev, padded, bad);
      if (n >= 0) atomicAdd(&base[n], 1);  // count
    }
  }
  __syncthreads();
  const long long seg0 = (long long)(t0 / d.chunk) * d.nseg() + bg * d.nblk;
  for (int i = threadIdx.x; i < nmax; i += kHistRows)  // reserve each list's range: count -> start
    if (base[i]) base[i] = seg_offset[seg0 + i] + atomicAdd(seg_cursor + seg0 + i, base[i]);
  __syncthreads();
  int prev = -1;
  bool padded = false, bad = false;
  for (int s = 0; s < d.top_k; ++s) {
    const int n = checked_block(row, s, t, prev, padded, bad);
    if (n >= 0) entries[base[n] + atomicAdd(&cur[n], 1)] = (t << 8) | s;
  }
}

// Dense lists: chunk c of block n holds the tokens t >= 128 n with t in the chunk, i.e. the range
// [max(128 n, c * chunk), min(S, (c+1) * chunk)).
__device__ __forceinline__ long long dense_first(const Dims& d, long long seg) {
  const long long n = seg % d.nblk, c = seg / d.nseg();
  const long long lo = (long long)c * d.chunk;
  return n * kBlock > lo ? n * kBlock : lo;
}
__device__ __forceinline__ long long list_len(const Dims& d, bool dense, const int* seg_count,
                                              long long seg) {
  if (dense) {
    const long long c = seg / d.nseg();
    long long hi = (c + 1) * (long long)d.chunk;
    if (hi > d.S) hi = d.S;
    const long long lo = dense_first(d, seg);
    return hi > lo ? hi - lo : 0;
  }
  return seg_count[seg];
}

// Work items of a list of c entries (c <= S < 2^31: 32-bit arithmetic, whose division is several
// times cheaper than the 64-bit one in the single-block scan)
__device__ __forceinline__ int items_of(int c, const ItemSpec& s) {
  const int tiles = (c + s.tile_tokens - 1) / s.tile_tokens;
  return (tiles + s.chunk_tiles - 1) / s.chunk_tiles * s.nsub;
}

// Exclusive scans over every list of three running sums (list lengths and the item counts of up
// to two item specs), in three passes: per-tile sums (a tile = kScanTile consecutive lists, 8
// per thread), an exclusive scan of the tile sums (one block), and the per-list offsets of
// each tile from its tile's offset.  The lists number up to a few million (one per sequence
// chunk, batch, proxy head and key block), so the work is spread over every SM.
constexpr int kScanThreads = 1024, kScanPer = 8, kScanTile = kScanThreads * kScanPer;

struct Sums3 {
  long long a, b, c;
};

__device__ __forceinline__ Sums3 list_sums(const Dims& d, bool dense, const int* seg_count,
                                           long long s, int nspecs, const ItemSpec& s0,
                                           const ItemSpec& s1) {
  const long long len = list_len(d, dense, seg_count, s);
  return Sums3{len, nspecs > 0 ? (long long)items_of((int)len, s0) : 0,
               nspecs > 1 ? (long long)items_of((int)len, s1) : 0};
}

// Exclusive scan of v over the block's kScanThreads threads; *total receives the block's sum.
__device__ Sums3 block_exclusive_scan(Sums3 v, Sums3* total) {
  __shared__ long long sh[3][kScanThreads];
  const int tid = threadIdx.x;
  sh[0][tid] = v.a;
  sh[1][tid] = v.b;
  sh[2][tid] = v.c;
  __syncthreads();
  for (int off = 1; off < kScanThreads; off <<= 1) {  // inclusive Hillis-Steele scan
    long long va = 0, vb = 0, vc = 0;
    if (tid >= off) {
      va = sh[0][tid - off];
      vb = sh[1][tid - off];
      vc = sh[2][tid - off];
    }
    __syncthreads();
    sh[0][tid] += va;
    sh[1][tid] += vb;
    sh[2][tid] += vc;
    __syncthreads();
  }
  const Sums3 r{sh[0][tid] - v.a, sh[1][tid] - v.b, sh[2][tid] - v.c};
  *total = Sums3{sh[0][kScanThreads - 1], sh[1][kScanThreads - 1], sh[2][kScanThreads - 1]};
  __syncthreads();  // sh may be reused by the caller's next scan
  return r;
}

__device__ __forceinline__ Sums3 thread_sums(const Dims& d, bool dense, const int* seg_count,
                                             long long lo, long long nseg, int nspecs,
                                             const ItemSpec& s0, const ItemSpec& s1) {
  Sums3 v{0, 0, 0};
  for (int k = 0; k < kScanPer; ++k) {
    if (lo + k >= nseg) break;
    const Sums3 x = list_sums(d, dense, seg_count, lo + k, nspecs, s0, s1);
    v.a += x.a;
    v.b += x.b;
    v.c += x.c;
  }
  return v;
}

// The same scan in one block, tile after tile with a running carry: for up to kScanSingle
// tiles, where the three dependent launches would cost more than the work.
constexpr int kScanSingle = 8;
__global__ void __launch_bounds__(kScanThreads) scan_single_kernel(Dims d, int dense, const int* __restrict__ seg_count,
                                                                   int* __restrict__ seg_offset, ItemSpec s0,
                                                                   ItemSpec s1, int nspecs, int* __restrict__ io0,
                                                                   int* __restrict__ io1, int* __restrict__ totals) {
  const long long nseg = d.nlist();
  Sums3 carry{0, 0, 0};
  for (long long base = 0; base < nseg; base += kScanTile) {
    const long long lo = base + (long long)threadIdx.x * kScanPer;
    Sums3 tot;
    const Sums3 ex = block_exclusive_scan(thread_sums(d, dense, seg_count, lo, nseg, nspecs, s0, s1), &tot);
    long long ra = carry.a + ex.a, rb = carry.b + ex.b, rc = carry.c + ex.c;
    for (int k = 0; k < kScanPer; ++k) {
      const long long s = lo + k;
      if (s >= nseg) break;
      const Sums3 x = list_sums(d, dense, seg_count, s, nspecs, s0, s1);
      if (seg_offset) seg_offset[s] = (int)ra;
      if (nspecs > 0) io0[s] = (int)rb;
      if (nspecs > 1) io1[s] = (int)rc;
      ra += x.a;
      rb += x.b;
      rc += x.c;
    }
    carry.a += tot.a;
    carry.b += tot.b;
    carry.c += tot.c;
  }
  if (threadIdx.x == 0) {
    if (seg_offset) seg_offset[nseg] = (int)carry.a;
    totals[0] = (int)carry.a;
    totals[1] = (int)carry.b;
    totals[2] = (int)carry.c;
  }
}

// pass 1: tile_sums[3 t + {0, 1, 2}] = the sums of tile t
__global__ void __launch_bounds__(kScanThreads) scan_tiles_kernel(Dims d, int dense, const int* __restrict__ seg_count,
                                                                  ItemSpec s0, ItemSpec s1, int nspecs,
                                                                  long long* __restrict__ tile_sums) {
  const long long nseg = d.nlist();
  const long long lo = blockIdx.x * (long long)kScanTile + (long long)threadIdx.x * kScanPer;
  Sums3 tot;
  block_exclusive_scan(thread_sums(d, dense, seg_count, lo, nseg, nspecs, s0, s1), &tot);
  if (threadIdx.x == 0) {
    tile_sums[3 * blockIdx.x + 0] = tot.a;
    tile_sums[3 * blockIdx.x + 1] = tot.b;
    tile_sums[3 * blockIdx.x + 2] = tot.c;
  }
}

// pass 2 (one block): exclusive scan of the tile sums in place; totals = the grand sums
__global__ void __launch_bounds__(kScanThreads) scan_tops_kernel(long long* __restrict__ tile_sums, int ntiles,
                                                                 int* __restrict__ totals) {
  Sums3 carry{0, 0, 0};
  for (int base = 0; base < ntiles; base += kScanThreads) {
    const int t = base + (int)threadIdx.x;
    Sums3 v{0, 0, 0};
    if (t < ntiles) v = Sums3{tile_sums[3 * t], tile_sums[3 * t + 1], tile_sums[3 * t + 2]};
    Sums3 tot;
    const Sums3 ex = block_exclusive_scan(v, &tot);
    if (t < ntiles) {
      tile_sums[3 * t] = carry.a + ex.a;
      tile_sums[3 * t + 1] = carry.b + ex.b;
      tile_sums[3 * t + 2] = carry.c + ex.c;
    }
    carry.a += tot.a;
    carry.b += tot.b;
    carry.c += tot.c;
  }
  if (threadIdx.x == 0) {
    totals[0] = (int)carry.a;
    totals[1] = (int)carry.b;
    totals[2] = (int)carry.c;
  }
}

// pass 3: per-list offsets (seg_offset[nseg] = the total list length)
__global__ void __launch_bounds__(kScanThreads) scan_write_kernel(Dims d, int dense, const int* __restrict__ seg_count,
                                                                  int* __restrict__ seg_offset, ItemSpec s0,
                                                                  ItemSpec s1, int nspecs, int* __restrict__ io0,
                                                                  int* __restrict__ io1,
                                                                  const long long* __restrict__ tile_offsets,
                                                                  const int* __restrict__ totals) {
  const long long nseg = d.nlist();
  const long long lo = blockIdx.x * (long long)kScanTile + (long long)threadIdx.x * kScanPer;
  Sums3 tot;
  const Sums3 ex = block_exclusive_scan(thread_sums(d, dense, seg_count, lo, nseg, nspecs, s0, s1), &tot);
  long long ra = tile_offsets[3 * blockIdx.x] + ex.a, rb = tile_offsets[3 * blockIdx.x + 1] + ex.b,
            rc = tile_offsets[3 * blockIdx.x + 2] + ex.c;
  for (int k = 0; k < kScanPer; ++k) {
    const long long s = lo + k;
    if (s >= nseg) break;
    const Sums3 x = list_sums(d, dense, seg_count, s, nspecs, s0, s1);
    if (seg_offset) seg_offset[s] = (int)ra;
    if (nspecs > 0) io0[s] = (int)rb;
    if (nspecs > 1) io1[s] = (int)rc;
    ra += x.a;
    rb += x.b;
    rc += x.c;
  }
  if (seg_offset && blockIdx.x == 0 && threadIdx.x == 0) seg_offset[nseg] = totals[0];
}

__global__ void items_kernel(Dims d, int dense, const int* __restrict__ seg_count,
                             const int* __restrict__ seg_offset, ItemSpec sp,
                             const int* __restrict__ item_offset, Item* __restrict__ items,
                             long long max_items, unsigned* status) {
  const long long nseg = d.nlist();
  const int per_item = sp.tile_tokens * sp.chunk_tiles;
  for (long long seg = blockIdx.x; seg < nseg; seg += gridDim.x) {  // a block per list in turn
    const int len = (int)list_len(d, dense, seg_count, seg);
    const int n_items = (len + per_item - 1) / per_item * sp.nsub;
    const long long base = item_offset[seg];
    const long long list0 = seg_offset ? seg_offset[seg] : 0;
    for (int i = threadIdx.x; i < n_items; i += blockDim.x) {
      const long long pos = base + i;
      if (pos >= max_items) {
        atomicOr(status, kStatusBadItems);
        continue;
      }
      const int first = i / sp.nsub * per_item;  // the attention groups of a run of tokens
      const int cnt = len - first < per_item ? len - first : per_item;  // are consecutive
      items[pos] = Item{(int)seg, first, cnt, (int)(list0 + first), i % sp.nsub};
    }
  }
}

// Row data of every list entry, in entry order, so the gradient passes read it with the entry
// instead of through its token: lpxe[e] = LSE_px(b, p, t(e)) * log2 e and, for the Gp = Hq / Hp
// query heads of proxy head p, emeta[e Gp + h] = {LSE(b, p Gp + h, t(e)) log2 e,
// D(b, t(e), p Gp + h)}.
__global__ void entry_meta_kernel(Dims d, const int* __restrict__ seg_count,
                                  const int* __restrict__ seg_offset, const int* __restrict__ entries,
                                  const float* __restrict__ lse_px, const float2* __restrict__ rowm,
                                  float* __restrict__ lpxe, float2* __restrict__ emeta) {
  // one block per list: the lists' lengths vary by orders of magnitude (a block every token
  // selects against a rarely chosen one), which the block scheduler balances
  const long long seg = blockIdx.x;
  const int len = (int)list_len(d, false, seg_count, seg);
  if (len == 0) return;
  const long long base = seg_offset[seg];
  const long long bg = (seg % d.nseg()) / d.nblk;  // b * Hp + g
  const long long b = bg / d.Hp, g = bg % d.Hp;
  const float* row = lse_px + bg * d.S;
  for (int k = threadIdx.x; k < len; k += blockDim.x) {
    const long long t = entries[base + k] >> 8;
    lpxe[base + k] = row[t] * kLog2e;
  }
  const int gp = d.Gp();
  const int n = len * gp;  // < 2^31: 32-bit index arithmetic
  for (int x = threadIdx.x; x < n; x += blockDim.x) {
    const int k = x / gp, h = x - k * gp;
    const long long t = entries[base + k] >> 8;
    emeta[base * gp + x] = rowm[((b * d.S + t) * d.Hq + g * gp + h)];
  }
}

__global__ void convert_kernel(const float4* __restrict__ src, uint2* __restrict__ dst, long long n4) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 v = src[i];
    dst[i] = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
  }
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

static int grid_for(long long work, int threads) {
  long long g = (work + threads - 1) / threads;
  const long long cap = (long long)num_sms() * 16;
  if (g > cap) g = cap;
  return g < 1 ? 1 : (int)g;
}

void launch_count(const Dims& d, const int32_t* idx, int* seg_count, unsigned* status,
                  cudaStream_t st) {
  const long long rows = (long long)d.B * d.Hp * d.S;
  if (d.nblk <= kHistBlocks)
    count_hist_kernel<<<(unsigned)(rows / kHistRows), kHistRows, 0, st>>>(d, idx, seg_count, status);
  else
    count_kernel<<<grid_for(rows, 256), 256, 0, st>>>(d, idx, seg_count, status);
}

long long scan_tiles(long long nlists) { return (nlists + kScanTile - 1) / kScanTile; }

int scan_kernels(long long nlists) { return scan_tiles(nlists) <= kScanSingle ? 1 : 3; }

void launch_scan(const Dims& d, bool dense, const int* seg_count, int* seg_offset,
                 const ItemSpec* specs, int nspecs, int* item_offset0, int* item_offset1,
                 int* totals, long long* tile_tmp, cudaStream_t st) {
  ItemSpec s0 = nspecs > 0 ? specs[0] : ItemSpec{1, 1, 1};
  ItemSpec s1 = nspecs > 1 ? specs[1] : ItemSpec{1, 1, 1};
  const int ntiles = (int)scan_tiles(d.nlist());
  if (ntiles <= kScanSingle) {
    scan_single_kernel<<<1, kScanThreads, 0, st>>>(d, dense ? 1 : 0, seg_count, seg_offset, s0, s1,
                                                   nspecs, item_offset0, item_offset1, totals);
    return;
  }
  scan_tiles_kernel<<<ntiles, kScanThreads, 0, st>>>(d, dense ? 1 : 0, seg_count, s0, s1, nspecs,
                                                     tile_tmp);
  scan_tops_kernel<<<1, kScanThreads, 0, st>>>(tile_tmp, ntiles, totals);
  scan_write_kernel<<<ntiles, kScanThreads, 0, st>>>(d, dense ? 1 : 0, seg_count, seg_offset, s0,
                                                     s1, nspecs, item_offset0, item_offset1,
                                                     tile_tmp, totals);
}

void launch_fill(const Dims& d, const int32_t* idx, const int* seg_offset, int* seg_cursor,
                 int* entries, unsigned* status, cudaStream_t st) {
  (void)status;
  const long long rows = (long long)d.B * d.Hp * d.S;
  if (d.nblk <= kHistBlocks)
    fill_hist_kernel<<<(unsigned)(rows / kHistRows), kHistRows, 0, st>>>(d, idx, seg_offset,
                                                                         seg_cursor, entries);
  else
    fill_kernel<<<grid_for(rows, 256), 256, 0, st>>>(d, idx, seg_offset, seg_cursor, entries);
}

void launch_items(const Dims& d, bool dense, const int* seg_count, const int* seg_offset,
                  const ItemSpec& spec, const int* item_offset, Item* items, long long max_items,
                  unsigned* status, cudaStream_t st) {
  items_kernel<<<grid_for(d.nlist(), 1), 128, 0, st>>>(d, dense ? 1 : 0, seg_count, seg_offset,
                                                       spec, item_offset, items, max_items, status);
}

void launch_entry_meta(const Dims& d, const int* seg_count, const int* seg_offset,
                       const int* entries, const float* lse_px, const float2* rowm, float* lpxe,
                       float2* emeta, cudaStream_t st) {
  entry_meta_kernel<<<(unsigned)d.nlist(), 256, 0, st>>>(d, seg_count, seg_offset, entries, lse_px,
                                                          rowm, lpxe, emeta);
}

void launch_convert(const float* src, void* dst, long long n, cudaStream_t st) {
  const long long n4 = n / 4;
  convert_kernel<<<grid_for(n4, 256), 256, 0, st>>>(reinterpret_cast<const float4*>(src),
                                                    reinterpret_cast<uint2*>(dst), n4);
}

}  // namespace msa
