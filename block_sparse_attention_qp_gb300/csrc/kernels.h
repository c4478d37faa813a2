// Internal interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace msa {

// Head mapping (the MSA group is the proxy head): proxy head p selects key blocks for its Hq / Hp
// query heads.  An attention group is a set of G query heads that share one selection row and
// one KV head: G = Hq / max(Hp, Hkv), and proxy head p has R = max(1, Hkv / Hp) of them,
// a = p R + r (r < R), on KV head kv_of(a).  Hp == Hkv: a = p = the GQA group, R = 1.
struct Dims {
  int B, S, Hq, Hkv, Hp, G, top_k, nblk;
  float scale;
  int chunk;   // token-list chunk: a list holds the tokens of one (b, p, n) in one chunk of the
  int nchunk;  // sequence [c * chunk, (c+1) * chunk); lists are ordered chunk-major
  int R = 1;   // attention groups per proxy head
  __host__ __device__ long long nseg() const { return (long long)B * Hp * nblk; }  // (b, p, n)
  __host__ __device__ long long nlist() const { return nseg() * nchunk; }           // (c, b, p, n)
  __host__ __device__ int kv_of(int a) const { return a / (Hp * R / Hkv); }
  __host__ __device__ int Gp() const { return G * R; }  // query heads per proxy head
};

// A unit of attention work: `count` tokens of list `seg` (= c * nseg + (b * Hp + p) * nblk + n)
// starting at list position `first`, for attention group p R + sub; `base` = the list's offset +
// first, i.e. the position of the item's first entry in the packed entry array.
struct Item {
  int seg, first, count, base, sub;
};

// Shape of one work list: tiles of `tile_tokens` tokens, `chunk_tiles` tiles per item, and
// `nsub` items (attention groups r = 0 .. nsub-1) for each such run of tokens.
struct ItemSpec {
  int tile_tokens, chunk_tiles, nsub;
};

// ---------------------------------------------------------------- index kernels (index.cu)
// Count block references per (c, b, g, n) list (validating every index against its row).
void launch_count(const Dims& d, const int32_t* idx, int* seg_count, unsigned* status,
                  cudaStream_t st);
// Exclusive scans: list offsets (sparse only) and item offsets for up to two item specs.
// dense: list lengths are the tokens t >= 128 n of the chunk instead of seg_count.
// tile_tmp: scan_tiles(d.nlist()) x 3 long longs of scratch.  scan_kernels: how many kernels
// one scan launches (one block for few lists, three passes over every SM otherwise).
long long scan_tiles(long long nlists);
int scan_kernels(long long nlists);
void launch_scan(const Dims& d, bool dense, const int* seg_count, int* seg_offset,
                 const ItemSpec* specs, int nspecs, int* item_offset0, int* item_offset1,
                 int* totals, long long* tile_tmp, cudaStream_t st);
// Scatter (t << 8 | slot) into the lists; order inside a list is unspecified.
void launch_fill(const Dims& d, const int32_t* idx, const int* seg_offset, int* seg_cursor,
                 int* entries, unsigned* status, cudaStream_t st);
void launch_items(const Dims& d, bool dense, const int* seg_count, const int* seg_offset,
                  const ItemSpec& spec, const int* item_offset, Item* items, long long max_items,
                  unsigned* status, cudaStream_t st);

// Row data of every entry e of the sparse lists, in entry order: lpxe[e] = LSE_px of e's token
// x log2(e); emeta[e Gp + h] = rowm of e's token and head g Gp + h.  (Dense lists need no copy:
// their tokens are consecutive, and the dense kernels read rowm and LSE_px by token.)
void launch_entry_meta(const Dims& d, const int* seg_count, const int* seg_offset,
                       const int* entries, const float* lse_px, const float2* rowm, float* lpxe,
                       float2* emeta, cudaStream_t st);

// ---------------------------------------------------------------- proxy top-k (topk.cu)
// Returns false if the TMA tensor maps could not be created (driver entry point missing).
bool launch_proxy_topk(const Dims& d, const void* qp, const void* kp, int32_t* idx,
                       unsigned* status, cudaStream_t st);
// Dense proxy normaliser (warmup): lse_px[(b Hp + g) S + t] = log sum_{j <= t} exp(scale qp.kp).
bool launch_proxy_lse_dense(const Dims& d, const void* qp, const void* kp, float* lse_px,
                            unsigned* status, cudaStream_t st);

// ---------------------------------------------------------------- forward (fwd.cu)
// Sparse main-attention partials (attn_fwd.cu): for every list entry (t, slot) and query head h
// of the group, the block's normalised output (bf16, opart[(t, h, slot)][128]) and its natural
// log-sum-exp (lpart).  Returns false for an unsupported group size or if the TMA tensor maps
// cannot be created.
// One pass takes the items [*item_lo, *item_hi) (NULL: 0 / all) -- the lists of a range of
// sequence chunks -- and indexes its partials from token pass_t0 ((b pass_tokens + t - pass_t0)
// Hq + h) top_k + slot.
bool launch_attn_fwd(const Dims& d, const void* q, const void* k, const void* v,
                     const int* seg_offset, const int* entries, const Item* items,
                     const int* n_items, long long max_items, const int* item_lo,
                     const int* item_hi, int pass_t0, int pass_tokens, void* opart, float* lpart,
                     unsigned* status, cudaStream_t st);
int fwd_item_tiles();  // 128-row tiles per sparse-forward work item
// Merges the partials of every (b, t, h) with t in [t0, t0 + tn) (partials indexed as the pass
// with pass_tokens = tp wrote them); a partial is valid iff its log-sum-exp is not NaN (the
// caller fills lpart with NaN bytes before the partial pass).
void launch_combine(const Dims& d, const void* opart, const float* lpart, void* o, float* lse,
                    int t0, int tn, int tp, cudaStream_t st);
// Dense causal forward of the warmup mode (dense_fwd.cu).  Returns false for an unsupported group
// size or if the TMA tensor maps cannot be created.
bool launch_dense_fwd(const Dims& d, const void* q, const void* k, const void* v, void* o,
                      float* lse, unsigned* status, cudaStream_t st);

// ---------------------------------------------------------------- backward (bwd.cu)
// rowm[(b S + t) Hq + h] = {LSE(b, h, t) log2 e, rowsum(dO * O)(b, t, h)}
void launch_bwd_rowdot(const Dims& d, const void* o, const void* dout, const float* lse,
                       float2* rowm, cudaStream_t st);
// Sparse proxy normaliser, first pass (attn_fwd.cu, proxy mode): lpx_part[((b S + t) Hp + g) top_k
// + slot] = log-sum-exp of scale qp.kp over the visible keys of that slot's block; slots no list
// entry reaches are left as they were (the caller fills lpx_part with NaN bytes first).
bool launch_proxy_lse_sparse(const Dims& d, const void* qp, const void* kp, const int* seg_offset,
                             const int* entries, const Item* items, const int* n_items,
                             long long max_items, float* lpx_part, unsigned* status,
                             cudaStream_t st);
// Second pass: lse_px[(b Hp + g) S + t] from the written (non-NaN) partials of each row.
void launch_proxy_lse_combine(const Dims& d, const float* lpx_part, float* lse_px, cudaStream_t st);

// Main-attention backward (dQ, dK, dV into fp32 accumulators) and the teacher pbar
// ([list entry - *entry_lo][128 keys] fp16) of one pass: the items [*item_lo, *item_hi) (NULL:
// 0 / all; entry_lo NULL: 0).  rowdata: {LSE log2 e, D} per list entry and head (emeta, sparse)
// or per query row (rowm [B, S, Hq], dense).  Returns false for an unsupported group size or if
// the TMA tensor maps cannot be created.
bool launch_attn_bwd(const Dims& d, bool dense, const void* q, const void* k, const void* v,
                     const void* dout, const float2* rowdata, const int* seg_offset,
                     const int* entries, const Item* items, const int* n_items, long long max_items,
                     const int* item_lo, const int* item_hi, const int* entry_lo,
                     float* dq_acc, float* dk_acc, float* dv_acc, void* pbar, unsigned* status,
                     cudaStream_t st);
// Proxy gradients (dQp, dKp into fp32 accumulators) of the KL term from pbar, scaled by kl_grad,
// or by *kl_grad_dev (read on the device) when that is not NULL.  kl_acc: NULL, or
// a zeroed double that receives sum over the visited (token, key) pairs of
// pbar (ln pbar - ln p_student), i.e. B S Hp times the KL value.
// lpx: LSE_px x log2 e per list entry (lpxe, sparse) or LSE_px per proxy row (lse_px
// [B, Hp, S], dense).
bool launch_proxy_bwd(const Dims& d, bool dense, const void* qp, const void* kp,
                      const float* lpx, const void* pbar, float kl_grad,
                      const float* kl_grad_dev, const int* seg_offset,
                      const int* entries, const Item* items, const int* n_items,
                      long long max_items, const int* item_lo, const int* item_hi,
                      const int* entry_lo, float* dqp_acc, float* dkp_acc, double* kl_acc,
                      unsigned* status, cudaStream_t st);  // one pass, as launch_attn_bwd
// kl_out[0] = kl_acc[0] / (B S Hp)  (one thread)
void launch_kl_finalize(const Dims& d, const double* kl_acc, float* kl_out, cudaStream_t st);
int bwd_item_tokens();   // tokens per fused-backward work item
int bwd_group_tokens();  // tokens per proxy-gradient flush group
void launch_convert(const float* src, void* dst, long long n, cudaStream_t st);

// ---------------------------------------------------------------- decode (decode.cu)
// One new token per sequence against its cache, in three launches: proxy block scores (scores
// [B, Hp, nblk] fp32), selection (block_idx [B, Hp, top_k]) and sparse attention (o [B, Hq, 128],
// lse [B, Hq]).
bool launch_decode_scores(const Dims& d, const void* qp, const void* kp_cache,
                          const int32_t* seq_len, float* scores, unsigned* status,
                          cudaStream_t st);  // false: the tensor map could not be made
void launch_decode_select(const Dims& d, const float* scores, const int32_t* seq_len,
                          int32_t* block_idx, cudaStream_t st);
bool launch_decode_attn(const Dims& d, const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* seq_len, const int32_t* block_idx, void* o, float* lse,
                        unsigned* status, cudaStream_t st);  // false: no tensor map

int num_sms();
void set_api_error(const char* what);

}  // namespace msa
