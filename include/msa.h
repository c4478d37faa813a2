/*
 * msa.h -- C ABI of libmsa.so: MiniMax Sparse Attention (MSA) training on one GB300 (sm_103a).
 *
 * The method (Flash-MSA blog, "About MSA"; MSA forum summary, "Architecture: two-stage
 * block-sparse attention"): causal GQA attention in which one proxy (index) query head per GQA
 * group, scored against one shared proxy key head, picks for every query the top-k 128-token key
 * blocks -- the query's own (local) block always among them -- and the main attention runs
 * exactly, with softmax, over the picked blocks only.  The proxy is trained by a KL loss towards
 * the group's mean main-attention distribution over the same tokens (blog, "KL Divergence Loss").
 *
 * Conventions shared by every entry point
 *   Tensors are dense, row-major, on the current CUDA device, caller-owned:
 *     q, o, dout, dq    [B, S, Hq,  128]  bf16
 *     k, v, dk, dv      [B, S, Hkv, 128]  bf16
 *     qp, dqp           [B, S, Hp,  128]  bf16   (proxy queries, one head per selection row)
 *     kp, dkp           [B, S, 1,   128]  bf16   (one proxy key head shared by every proxy head)
 *     lse               [B, Hq, S]        fp32   natural-log sum of exp of the scaled scores
 *     block_idx         [B, Hp, S, top_k] int32  selected key blocks per (b, proxy head, token),
 *                                                ascending, padded with -1 when fewer than
 *                                                top_k blocks are visible
 *   Head mapping (blog, "Context parallelism" point 1: an MSA group is the query heads assigned
 *   to one proxy head; "Note about scheduler requiring proxy heads >= KV heads": more KV heads
 *   than proxy heads inverts that mapping; the top-k sweep footnote runs 4 proxy heads over 2 KV
 *   heads): query head h reads KV head h / (Hq / Hkv) and takes the selection of proxy head
 *   h / (Hq / Hp).  Hq must be a multiple of Hkv and of Hp, and one
 *   of Hp, Hkv a multiple of the other.  The KL teacher of proxy head p is the mean main
 *   softmax of its Hq / Hp query heads.  Key j is visible to token t iff j <= t.
 *   Every pointer must be 16-byte aligned.  Supported: head dim 128, block 128 (blog / package
 *   caveat 1), S % 128 == 0, 1 <= top_k <= 64, and Hq / max(Hp, Hkv) -- the query heads that
 *   share both one KV head and one selection row -- in {1, 2, 4, 8, 16} for the forward ops and
 *   {4, 8, 16} for the backward ops (the warmup forward, which has no selection: Hq / Hkv).
 *   Other shapes return MSA_ERR_UNSUPPORTED.
 *   `workspace` is caller-owned device memory of at least msa_workspace_size() bytes for the
 *   same op and shape; the library allocates no device memory.  The first 256 bytes hold a device status
 *   word (see msa_device_status) and the work-item counters of the persistent kernels (reset on
 *   the stream before each launch).  Calls sharing one workspace must not overlap on the GPU.
 *   `stream` is a cudaStream_t (NULL = legacy default stream); all work is asynchronous and
 *   ordered on it.  The backward ops run two independent memory-bound steps (zeroing of their
 *   accumulators with the row data D; the bf16 conversion of dQ, dK, dV) on a side stream that the
 *   library creates once per host thread and device, forked from `stream` with an event and
 *   joined back into it before the call returns: the call's work still completes in `stream`'s
 *   order, and a CUDA graph capture of the call stays closed.
 *   Return value: an msa_status code.  Argument errors are detected on the host before any
 *   launch; MSA_ERR_CUDA reports a launch or runtime error (msa_last_error() gives the text).
 *   No entry point synchronises the device except msa_device_status.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MSA_API __attribute__((visibility("default")))
#else
#define MSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct msa_shape {
  int32_t B;      /* batch */
  int32_t S;      /* sequence length, multiple of 128 */
  int32_t Hq;     /* main query heads */
  int32_t Hkv;    /* main key/value heads (GQA groups) */
  int32_t Hp;     /* proxy query heads (see the head mapping above) */
  int32_t D;      /* head dim, must be 128 */
  int32_t top_k;  /* selected blocks per query, local block included (ignored by warmup ops) */
  float scale;    /* softmax scale of both attentions, usually 128^-0.5 */
} msa_shape_t;

enum msa_status {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1, /* null / misaligned pointer, non-positive size */
  MSA_ERR_UNSUPPORTED = 2, /* D != 128, S % 128 != 0, head counts, group size or top_k */
  MSA_ERR_WORKSPACE = 3,   /* workspace too small */
  MSA_ERR_CUDA = 4         /* CUDA launch / runtime error */
};

enum msa_op {
  MSA_OP_FORWARD = 0,
  MSA_OP_BACKWARD = 1,
  MSA_OP_WARMUP_FORWARD = 2,
  MSA_OP_WARMUP_BACKWARD = 3,
  MSA_OP_DECODE = 4
};

/* Bits of the device status word. */
#define MSA_DEVICE_BAD_INDEX 1u /* a given block index was out of range or not ascending */
#define MSA_DEVICE_BAD_ITEMS 2u /* internal work list overflow (a library bug) */
#define MSA_DEVICE_TIMEOUT 4u   /* a bounded device-side wait gave up */
#define MSA_DEVICE_INTERNAL 8u  /* a kernel's internal layout check failed (a library bug) */
/* With MSA_DEVICE_TIMEOUT set, the 32-bit word at byte offset 64 of the workspace may name the
 * first wait that gave up (a nonzero place number of the kernel that set it); diagnostic only. */

/* Bytes of workspace `op` needs for `shape` (0 if the shape is unsupported). */
MSA_API size_t msa_workspace_size(const msa_shape_t* shape, int op);

/*
 * Sparse forward (blog, "Forward": proxy attention, then sparse main attention; package usage
 * `flash_msa_func`).
 *   1. unless indices_given: proxy scores Qp.Kp^T per group, causal max-pool per 128-key block,
 *      the local block forced in, top-k with ties going to the lower block index
 *      (blog "Proxy attention") -> block_idx (written);
 *   2. exact softmax attention of every query head over the key blocks of its group in
 *      block_idx (blog "Main attention"; forum summary "Architecture") -> o, lse.
 * indices_given != 0: block_idx is an input (for instance the cached indices of an earlier
 * call); invalid entries are skipped and flagged with MSA_DEVICE_BAD_INDEX.
 * Workspace: the per-(token, head, slot) partial outputs of step 2 are produced and merged in
 * passes over consecutive sequence chunks.  msa_workspace_size sizes them for passes of at most
 * 8 GiB of partials; a larger workspace_bytes gives fewer passes, a smaller one more (down to one
 * chunk per pass; below that MSA_ERR_WORKSPACE).  The results do not depend on the passes.
 */
MSA_API int msa_forward(const msa_shape_t* shape, const void* q, const void* k, const void* v,
                const void* qp, const void* kp, int32_t* block_idx, int indices_given, void* o,
                float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Sparse backward (blog, "Backward" and "KL Divergence Loss").  From the cached block_idx it
 * inverts the block map, recomputes the proxy normaliser over the selected tokens, and in one
 * fused pass per (key block, group) recomputes the main and proxy probabilities and emits
 *   dq, dk, dv  of  sum(o * dout)                     (teacher detached: no KL term here)
 *   dqp, dkp    of  kl_grad * L_KL,  L_KL = mean over (b, t, proxy head) of
 *               KL(teacher || student), teacher = mean over the proxy head's Hq / Hp query
 *               heads of the main softmax (stop-gradient),
 *               student = softmax(scale * qp . kp) over the same tokens; the score gradient is
 *               kl_grad / (B*S*Hp) * (p_student - p_teacher)  (blog, "KL Divergence Loss").
 * o and lse are the outputs of msa_forward for the same inputs.  kl_grad is the incoming
 * gradient of the (zero) KL placeholder the forward returns (package usage note), usually 1.
 * Workspace: the teacher rows (one fp16 row of 128 keys per list entry) live for one pass of
 * consecutive sequence chunks at a time (attn_bwd writes them, the proxy gradients read them);
 * msa_workspace_size sizes a pass for at most 8 GiB of them, a larger workspace_bytes gives fewer
 * passes and a smaller one more (down to one chunk per pass; below that MSA_ERR_WORKSPACE).
 * kl_grad_dev: NULL, or a device pointer to one float that is used instead of kl_grad, read by
 * the kernel (an autograd backward can pass the placeholder's incoming gradient tensor without a
 * host synchronisation).
 * kl_out: NULL, or a device pointer to one float that receives the KL value L_KL itself (not
 * scaled by kl_grad).  The gradients never need it (blog, "KL Divergence Loss": the proxy
 * gradient is p_student - p_teacher), so it is computed only on request -- for logging every n
 * steps -- from the teacher and student probabilities the proxy-gradient pass already holds, at
 * the cost of one logarithm per selected (token, key) pair (package caveat 2: the reference
 * package does not return it at all).
 */
MSA_API int msa_backward(const msa_shape_t* shape, const void* q, const void* k, const void* v,
                 const void* qp, const void* kp, const void* o, const float* lse,
                 const void* dout, const int32_t* block_idx, float kl_grad,
                 const float* kl_grad_dev, void* dq, void* dk, void* dv, void* dqp, void* dkp,
                 float* kl_out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Warmup forward (blog, "Warmup kernels"): dense causal GQA attention, no proxy pass.
 * Writes o and lse.  top_k is ignored.
 */
MSA_API int msa_warmup_forward(const msa_shape_t* shape, const void* q, const void* k, const void* v,
                       void* o, float* lse, void* workspace, size_t workspace_bytes,
                       void* stream);

/*
 * Warmup backward (blog, "Warmup kernels"): the proxy normaliser over the full causal prefix,
 * then the fused main + proxy backward with every visible key in the key set.  Same outputs
 * (kl_grad_dev and kl_out included) and KL definition as msa_backward.  top_k is ignored.
 * Workspace: the teacher rows live for one pass of consecutive dense lists at a time (a pass may
 * end inside a sequence chunk), so the workspace does not grow with the square of S beyond them:
 * msa_workspace_size sizes a pass for at most 8 GiB of teacher rows, a larger workspace_bytes
 * gives fewer passes and a smaller one more (down to one list -- at most one chunk of tokens --
 * per pass; below that MSA_ERR_WORKSPACE).  The results do not depend on the passes beyond the
 * order of the fp32 gradient reductions.
 */
MSA_API int msa_warmup_backward(const msa_shape_t* shape, const void* q, const void* k, const void* v,
                        const void* qp, const void* kp, const void* o, const float* lse,
                        const void* dout, float kl_grad, const float* kl_grad_dev, void* dq,
                        void* dk, void* dv, void* dqp, void* dkp, float* kl_out, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * Decode step of MSA inference (forum summary, "GPU kernel co-design", deployment setting
 * B = 128, k = 16; the prefill is msa_forward).  One new token per sequence b, at position
 * t_b = seq_len[b] - 1 of its caches, whose K, V and proxy key rows must already hold it:
 *   q         [B, Hq, 128]  bf16   the new tokens' queries
 *   qp        [B, Hp, 128]  bf16   their proxy queries
 *   k_cache, v_cache [B, S, Hkv, 128] bf16, kp_cache [B, S, 128] bf16: caches of capacity S
 *             (shape->S, a multiple of 128); rows after t_b are never read
 *   seq_len   [B] int32 device array, 1 <= seq_len[b] <= S (other values: the row is skipped and
 *             MSA_DEVICE_BAD_INDEX set)
 * Writes block_idx [B, Hp, top_k] (the selection of the new token: the local block t_b / 128 and
 * the best top_k - 1 earlier blocks by raw proxy score, ties to the lower block, ascending, -1
 * padded), o [B, Hq, 128] bf16 and lse [B, Hq] fp32 -- the same values as row t_b of msa_forward
 * on the whole sequence.  Head mapping and limits as for msa_forward, with Hp <= 32.  Workspace:
 * msa_workspace_size(shape, MSA_OP_DECODE).
 */
MSA_API int msa_decode(const msa_shape_t* shape, const void* q, const void* qp,
                       const void* k_cache, const void* v_cache, const void* kp_cache,
                       const int32_t* seq_len, int32_t* block_idx, void* o, float* lse,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * Reads (and clears) the device status word of `workspace` after the work queued on `stream`
 * finishes; this synchronises `stream`.  *flags receives MSA_DEVICE_* bits (0 = clean).
 */
MSA_API int msa_device_status(void* workspace, unsigned* flags, void* stream);

/*
 * Measurement aids (not part of the method).  msa_profile_begin() makes every later call record
 * a CUDA event pair around each kernel it launches, on the launch stream.  msa_profile_end()
 * waits for those events, writes one line per kernel name -- "<name> <launches> <total_ms>\n" --
 * into buf (NUL-terminated, truncated to len) and stops recording.  msa_launch_count() returns
 * the number of kernels this library has launched since it was loaded.
 */
MSA_API int msa_profile_begin(void);
MSA_API int msa_profile_end(char* buf, size_t len);
MSA_API long long msa_launch_count(void);

/*
 * Allocation-free variant of msa_forward (the method's pages have no counterpart; this is an
 * integration aid).  Some callers cannot allocate device memory where they call the forward --
 * for example a C layer embedded in a framework whose allocator it cannot reach, or code running
 * while a sequence of launches is being recorded for replay, where allocating is not allowed.
 * This entry point needs no workspace: it uses a fixed scratch array of 64 MiB (67108864 bytes)
 * that lives in device memory for as long as the library is loaded, one per GPU that loads it.  Arguments and results are those of msa_forward; inputs and outputs are still
 * the caller's.  Shapes whose forward workspace exceeds the array are rejected with
 * MSA_ERR_WORKSPACE before any launch.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress), so make that first call before any stream capture.  Every call
 * on a device shares the one array and it keeps the last call's contents: the call re-initialises
 * what must start at zero itself, but calls that overlap on the GPU (different streams without
 * ordering) race on it and must be serialised by the caller.
 */
MSA_API int msa_forward_noalloc(const msa_shape_t* shape, const void* q, const void* k,
                                const void* v, const void* qp, const void* kp, int32_t* block_idx,
                                int indices_given, void* o, float* lse, void* stream);

/*
 * Device status word of the fixed scratch array that msa_forward_noalloc uses on the current
 * device: same bits and behaviour as msa_device_status (reads and clears the word once the work
 * queued on `stream` has finished; synchronises `stream`).  Callers of msa_forward_noalloc have no
 * workspace pointer to pass to msa_device_status, so this is how they learn that given block
 * indices were skipped as invalid (MSA_DEVICE_BAD_INDEX) or that a bounded wait gave up.  Every
 * call of msa_forward_noalloc on a device clears the word before it launches, so read it after
 * each call whose result matters.
 */
MSA_API int msa_forward_noalloc_status(unsigned* flags, void* stream);

/*
 * Failure-detection self-test (not part of the method).  Launches one block on `stream` whose
 * thread waits on a shared-memory mbarrier that nothing arrives at, through the same bounded wait
 * every kernel of the library uses; after limit_us microseconds (1 .. 1000000) the wait gives up
 * and sets MSA_DEVICE_TIMEOUT in the status word of `workspace` (any workspace of this library, or
 * 256 zeroed, 16-byte aligned device bytes).  Read it with msa_device_status.  Returns
 * MSA_ERR_INVALID_ARG for a null or misaligned workspace or a limit out of range.
 */
MSA_API int msa_selftest_wait_timeout(void* workspace, unsigned limit_us, void* stream);

/* Static text for a status code. */
MSA_API const char* msa_status_string(int status);

/* Detail of the last error on the calling thread ("" if none). */
MSA_API const char* msa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
