// C ABI of libmsa.so (declared in include/msa.h): argument validation, workspace carving and
// the launch sequence of every entry point.  All work is ordered on the caller's stream; the
// backward runs two pieces of independent HBM-bound work on a side stream that it forks from and
// joins back into the caller's stream (see Branch).
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/msa.h"
#include "common.cuh"
#include "kernels.h"

namespace msa {
namespace {

thread_local char g_err[512] = "";

void set_err(const char* what) {
  snprintf(g_err, sizeof(g_err), "%s", what);
}

int cuda_fail(const char* where) {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return MSA_OK;
  snprintf(g_err, sizeof(g_err), "%s: %s", where, cudaGetErrorString(e));
  return MSA_ERR_CUDA;
}

// ---- launch accounting and optional per-kernel event timing
std::atomic<long long> g_launches{0};
std::mutex g_prof_mu;
bool g_prof_on = false;
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pooled_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Runs `launch` (which issues `kernels` kernels on st, one unless stated), counting them and
// timing them together if enabled.
template <typename F>
void timed(const char* name, cudaStream_t st, F&& launch, int kernels = 1) {
  g_launches.fetch_add(kernels, std::memory_order_relaxed);
  if (!g_prof_on) {
    launch();
    return;
  }
  std::lock_guard<std::mutex> lk(g_prof_mu);
  ProfRec r{name, pooled_event(), pooled_event()};
  cudaEventRecord(r.a, st);
  launch();
  cudaEventRecord(r.b, st);
  g_prof.push_back(r);
}

// ---- a second stream for work that does not depend on the work queued beside it
// One per host thread and device, made on first use and kept for the life of the process.
struct Side {
  cudaStream_t s = nullptr;
  cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
  bool ready = false, failed = false;
};

Side* side_stream() {
  constexpr int kMaxDev = 64;
  thread_local Side sides[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return nullptr;
  }
  Side& x = sides[dev];
  if (!x.ready && !x.failed) {
    if (cudaStreamCreateWithFlags(&x.s, cudaStreamNonBlocking) == cudaSuccess &&
        cudaEventCreateWithFlags(&x.fork_ev, cudaEventDisableTiming) == cudaSuccess &&
        cudaEventCreateWithFlags(&x.join_ev, cudaEventDisableTiming) == cudaSuccess) {
      x.ready = true;
    } else {
      x.failed = true;
      cudaGetLastError();
    }
  }
  return x.ready ? &x : nullptr;
}

// A branch off the caller's stream: on construction the side stream waits for everything queued
// on the caller's stream so far; work queued on aux() then runs beside what the caller's stream
// does next, until join() (or the destructor, on every return path) puts the caller's stream
// behind it.  A call therefore stays ordered as a whole on the caller's stream, and a CUDA graph
// capture of it stays closed.  At most one branch is open at a time per host thread.  Without a
// side stream (its creation failed) aux() is the caller's stream and the work runs in order.
class Branch {
 public:
  explicit Branch(cudaStream_t main) : main_(main), side_(side_stream()) {
    if (side_) {
      cudaEventRecord(side_->fork_ev, main_);
      cudaStreamWaitEvent(side_->s, side_->fork_ev, 0);
    }
  }
  Branch(const Branch&) = delete;
  Branch& operator=(const Branch&) = delete;
  ~Branch() { join(); }
  cudaStream_t aux() const { return side_ ? side_->s : main_; }
  void join() {
    if (side_ && !joined_) {
      cudaEventRecord(side_->join_ev, side_->s);
      cudaStreamWaitEvent(main_, side_->join_ev, 0);
    }
    joined_ = true;
  }

 private:
  cudaStream_t main_;
  Side* side_;
  bool joined_ = false;
};

constexpr size_t kAlign = 256;

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Workspace layout of one op.  Offsets are bytes from the workspace base; 0 size = absent.
struct Plan {
  size_t status = 0, totals = 0, seg_count = 0, seg_offset = 0, seg_cursor = 0, entries = 0;
  size_t io0 = 0, io1 = 0, items0 = 0, items1 = 0;
  size_t opart = 0, lpart = 0, lpx_part = 0, lse_px = 0, lpxe = 0, rowm = 0, emeta = 0, pbar = 0;
  size_t dq = 0, dk = 0, dv = 0, dqp = 0, dkp = 0, scores = 0, scan = 0;
  size_t bytes = 0;
  long long max0 = 0, max1 = 0;
  ItemSpec spec0{1, 1}, spec1{1, 1};
  int pass_chunks = 1;  // forward: sequence chunks per pass of the partial outputs; backward:
                        // per pass of the teacher rows
  // warmup backward: its teacher passes as list boundaries (cuts[i] .. cuts[i+1], chunk-major
  // list numbers) and the most entries any of them holds
  std::vector<long long> cuts;
  long long pass_ent = 0;
};

struct Carver {
  size_t off = 0;
  size_t take(size_t n) {
    const size_t at = off;
    off += up(n);
    return at;
  }
};

long long dense_entries(const Dims& d) {  // sum over blocks of S - 128 n, per (b, g)
  return (long long)d.B * d.Hp * ((long long)d.S * d.nblk - (long long)kBlock * d.nblk * (d.nblk - 1) / 2);
}

long long max_items(long long entries, const Dims& d, const ItemSpec& s) {
  return (entries / ((long long)s.tile_tokens * s.chunk_tiles) + d.nlist()) * s.nsub + 1;
}

// Sequence chunk of the backward's token lists: the dQ rows one chunk contributes for one proxy
// head (chunk x Gp heads x 128 x fp32) are kept to <= 32 MB, so that most of them (and the chunk's
// Q and dO rows) stay resident in L2 while the work items of that chunk and group run.  Smaller
// chunks cut the lists into more, shorter items (more partly filled tiles and K / V loads): on
// GB300 at S = 64K, G = 8 (about 256 entries per sparse list at 32 MB) the backward was fastest at
// 32 MB among 16, 32, 64 and 128 MB, while at S = 1M, G = 4 (32 entries per list at 32 MB) 64 MB
// was 28 % faster.  So sparse lists shorter than 128 entries on average (a list of one chunk,
// proxy head and block holds about chunk x top_k x 128 / S entries) double the chunk, up to 64 MB.
int bwd_chunk(const Dims& d, bool sparse) {
  int c = kBlock;
  while ((long long)c * 2 * d.Gp() * kD * 4 <= (32ll << 20) && c * 2 <= d.S) c *= 2;
  if (sparse)
    while ((long long)c * d.top_k * kBlock < 128ll * d.S && c * 2 <= d.S &&
           (long long)c * 2 * d.Gp() * kD * 4 <= (64ll << 20))
      c *= 2;
  return c;
}

// Sequence chunk of the forward's token lists: one chunk's query rows of one proxy head
// (chunk x Gp heads x 128 x bf16) are kept to <= 16 MB, so the up to top_k reads of every query row
// (one per selected block) hit L2 while the items of that chunk and group run.  As in the
// backward, lists shorter than 128 entries on average leave most gathered tiles partly filled, so
// they double the chunk, up to 64 MB: on GB300 at S = 1M with 4 heads per group (16 entries per
// list at 16 MB) attn_fwd took 46.5 ms at 16 MB, 36.3 at 32 MB and 32.3 at 64 MB, while at
// S = 64K (256 entries per list) 32 and 64 MB were 0.5 and 2 % slower than 16 MB.
int fwd_chunk(const Dims& d) {
  int c = kBlock;
  while ((long long)c * 2 * d.Gp() * kD * 2 <= (16ll << 20) && c * 2 <= d.S) c *= 2;
  while ((long long)c * d.top_k * kBlock < 128ll * d.S && c * 2 <= d.S &&
         (long long)c * 2 * d.Gp() * kD * 2 <= (64ll << 20))
    c *= 2;
  return c;
}

Dims with_chunk(Dims d, int chunk) {
  d.chunk = chunk;
  d.nchunk = (d.S + chunk - 1) / chunk;
  return d;
}

// The sparse forward's partial outputs (bf16 O and fp32 log-sum-exp per token, head and slot)
// are produced and merged in passes over consecutive sequence chunks, so that they need not be
// held for the whole sequence at once: by default a pass holds at most kFwdPartialBudget bytes of
// them (one chunk at least).
constexpr size_t kFwdPartialBudget = 8ull << 30;

int pass_tokens(const Dims& d, int pass_chunks) {
  const long long t = (long long)pass_chunks * d.chunk;
  return (int)(t < d.S ? t : d.S);
}

int default_pass_chunks(const Dims& d) {
  const size_t per_chunk = (size_t)d.B * d.chunk * d.Hq * d.top_k * (kD * sizeof(bf16) + sizeof(float));
  const long long fit = (long long)(kFwdPartialBudget / per_chunk);
  return (int)(fit < 1 ? 1 : fit > d.nchunk ? d.nchunk : fit);
}

// The backward's teacher rows (fp16, one per list entry) likewise live for one pass at a time:
// attn_bwd writes them and proxy_bwd reads them, pass by pass.  A pass holds at most
// kBwdTeacherBudget bytes of them: consecutive sequence chunks of the sparse lists (one chunk at
// least), a run of consecutive dense lists in the warmup backward (one list at least).
constexpr size_t kBwdTeacherBudget = 8ull << 30;

// List entries of the chunks [c0, c1) of the sparse lists: the most there can be (top_k per token
// and proxy head).
long long pass_entries(const Dims& d, int c0, int c1) {
  const long long lo = (long long)c0 * d.chunk;
  const long long hi = (long long)c1 * d.chunk < d.S ? (long long)c1 * d.chunk : d.S;
  return (long long)d.B * d.Hp * (hi - lo) * d.top_k;
}

// The largest entry count of any pass of `pc` chunks.
long long max_pass_entries(const Dims& d, int pc) {
  long long m = 0;
  for (int c0 = 0; c0 < d.nchunk; c0 += pc) {
    const long long e = pass_entries(d, c0, c0 + pc < d.nchunk ? c0 + pc : d.nchunk);
    if (e > m) m = e;
  }
  return m;
}

// Entries of dense list `seg` (chunk-major number): the chunk's tokens t >= 128 n.
long long dense_list_len(const Dims& d, long long seg) {
  const long long c = seg / d.nseg(), n = seg % d.nblk;
  const long long a = c * d.chunk, z = a + d.chunk < d.S ? a + d.chunk : d.S;
  const long long lo = n * kBlock > a ? n * kBlock : a;
  return z > lo ? z - lo : 0;
}

// The warmup backward's teacher passes: runs of consecutive dense lists (a pass may end inside a
// sequence chunk) of about equal size, each holding at most `budget` entries unless one list
// alone holds more (then that list is a pass).  Returns the boundaries; *most = the largest pass.
std::vector<long long> dense_cuts(const Dims& d, long long budget, long long* most) {
  const long long total = dense_entries(d);
  if (budget < 1) budget = 1;
  const long long np = (total + budget - 1) / budget;
  const long long target = np > 1 ? (total + np - 1) / np : total;
  std::vector<long long> cuts{0};
  long long acc = 0, mx = 0;
  for (long long seg = 0; seg < d.nlist(); ++seg) {
    const long long len = dense_list_len(d, seg);
    if (acc > 0 && acc + len > target) {
      cuts.push_back(seg);
      mx = acc > mx ? acc : mx;
      acc = 0;
    }
    acc += len;
  }
  cuts.push_back(d.nlist());
  *most = acc > mx ? acc : mx;
  return cuts;
}

int bwd_pass_chunks(const Dims& d) {
  int pc = d.nchunk;
  while (pc > 1 && (size_t)max_pass_entries(d, pc) * kBlock * 2 > kBwdTeacherBudget) --pc;
  return pc;
}

// pass_chunks: chunks per pass (0: the default); dense_budget: entries per warmup-backward teacher
// pass (0: the default)
Plan make_plan(const Dims& d, int op, int pass_chunks = 0, long long dense_budget = 0) {
  Plan p;
  Carver c;
  const long long nseg = d.nlist();
  const long long rows_q = (long long)d.B * d.S * d.Hq;
  const long long rows_kv = (long long)d.B * d.S * d.Hkv;
  const long long rows_p = (long long)d.B * d.S * d.Hp;
  const long long rows_kp = (long long)d.B * d.S;
  const long long sparse_ent = rows_p * d.top_k;
  const int TT = kBlock / d.G;
  p.status = c.take(256);
  p.totals = c.take(4 * sizeof(int));
  if (op == MSA_OP_FORWARD || op == MSA_OP_BACKWARD || op == MSA_OP_WARMUP_BACKWARD)
    p.scan = c.take(scan_tiles(nseg) * 3 * sizeof(long long));
  if (op == MSA_OP_FORWARD || op == MSA_OP_BACKWARD) {
    p.seg_count = c.take(nseg * sizeof(int));
    p.seg_offset = c.take((nseg + 1) * sizeof(int));
    p.seg_cursor = c.take(nseg * sizeof(int));
    p.entries = c.take(sparse_ent * sizeof(int));
  }
  if (op == MSA_OP_FORWARD) {
    p.spec0 = ItemSpec{TT, fwd_item_tiles(), d.R};
    p.max0 = max_items(sparse_ent, d, p.spec0);
    p.io0 = c.take(nseg * sizeof(int));
    p.items0 = c.take(p.max0 * sizeof(Item));
    p.pass_chunks = pass_chunks > 0 ? pass_chunks : default_pass_chunks(d);
    const long long rows_pass = (long long)d.B * pass_tokens(d, p.pass_chunks) * d.Hq;
    p.opart = c.take((size_t)rows_pass * d.top_k * kD * sizeof(bf16));
    p.lpart = c.take((size_t)rows_pass * d.top_k * sizeof(float));
  }
  if (op == MSA_OP_BACKWARD || op == MSA_OP_WARMUP_BACKWARD) {
    const bool dense = op == MSA_OP_WARMUP_BACKWARD;
    const long long ent = dense ? dense_entries(d) : sparse_ent;
    // one item per attention group (the proxy gradient kernel takes those with sub == 0)
    const ItemSpec fused{bwd_group_tokens(), bwd_item_tokens() / bwd_group_tokens(), d.R};
    if (dense) {
      p.spec0 = fused;
      p.max0 = max_items(ent, d, p.spec0);
      p.seg_offset = c.take((nseg + 1) * sizeof(int));
      p.io0 = c.take(nseg * sizeof(int));
      p.items0 = c.take(p.max0 * sizeof(Item));
    } else {
      p.spec0 = ItemSpec{kBlock, fwd_item_tiles(), 1};  // proxy normaliser items (128-token tiles)
      p.spec1 = fused;
      p.max0 = max_items(ent, d, p.spec0);
      p.max1 = max_items(ent, d, p.spec1);
      p.io0 = c.take(nseg * sizeof(int));
      p.io1 = c.take(nseg * sizeof(int));
      p.items0 = c.take(p.max0 * sizeof(Item));
      p.items1 = c.take(p.max1 * sizeof(Item));
      p.lpx_part = c.take((size_t)rows_p * d.top_k * sizeof(float));
    }
    p.lse_px = c.take((size_t)rows_p * sizeof(float));
    p.rowm = c.take((size_t)rows_q * sizeof(float2));  // {LSE log2 e, D} per query row
    if (dense) {
      p.cuts = dense_cuts(d, dense_budget > 0 ? dense_budget : (long long)(kBwdTeacherBudget / (kBlock * 2)),
                          &p.pass_ent);
    } else {
      p.pass_chunks = pass_chunks > 0 ? pass_chunks : bwd_pass_chunks(d);
      p.pass_ent = max_pass_entries(d, p.pass_chunks);
    }
    p.pbar = c.take((size_t)p.pass_ent * kBlock * sizeof(uint16_t));  // teacher rows (fp16) of a pass
    if (!dense) {  // dense lists' tokens are consecutive: their row data is read by token
      p.lpxe = c.take((size_t)ent * sizeof(float));            // proxy log-normaliser per entry
      p.emeta = c.take((size_t)ent * d.Gp() * sizeof(float2));  // rowm per entry and query head
    }
    p.dq = c.take((size_t)rows_q * kD * sizeof(float));
    p.dk = c.take((size_t)rows_kv * kD * sizeof(float));
    p.dv = c.take((size_t)rows_kv * kD * sizeof(float));
    p.dqp = c.take((size_t)rows_p * kD * sizeof(float));
    p.dkp = c.take((size_t)rows_kp * kD * sizeof(float));
  }
  if (op == MSA_OP_DECODE) p.scores = c.take((size_t)d.B * d.Hp * d.nblk * sizeof(float));
  p.bytes = c.off;
  return p;
}

// The plan for a call with `bytes` of workspace: passes of the default size, or of as many
// sequence chunks as the workspace holds (more or fewer).  The caller checks that it fits.
Plan plan_for(const Dims& d, int op, size_t bytes) {
  Plan p = make_plan(d, op);
  if (op == MSA_OP_WARMUP_BACKWARD) {  // teacher passes sized by entries: all the room left
    const size_t fixed = p.bytes - up((size_t)p.pass_ent * kBlock * 2);
    if (bytes == p.bytes || bytes <= fixed) return p;  // (too small: the caller reports it)
    long long budget = (long long)((bytes - fixed) / (kBlock * 2));
    if (budget > dense_entries(d)) budget = dense_entries(d);
    const Plan q = make_plan(d, op, 0, budget);
    return q.bytes <= bytes ? q : p;
  }
  int pc = p.pass_chunks;
  if (bytes >= p.bytes) {
    while (pc < d.nchunk && make_plan(d, op, pc + 1).bytes <= bytes) ++pc;
  } else {
    while (pc > 1 && make_plan(d, op, pc).bytes > bytes) --pc;
  }
  return pc != p.pass_chunks ? make_plan(d, op, pc) : p;
}

// Shape checks shared by every op.  Returns MSA_OK or an error code (message set).
int check_shape(const msa_shape_t* s, int op, Dims* out) {
  if (!s) {
    set_err("shape is null");
    return MSA_ERR_INVALID_ARG;
  }
  if (s->B < 1 || s->S < 1 || s->Hq < 1 || s->Hkv < 1 || s->Hp < 1) {
    set_err("B, S, Hq, Hkv and Hp must be positive");
    return MSA_ERR_INVALID_ARG;
  }
  if (!(s->scale > 0.f)) {
    set_err("scale must be positive and finite");
    return MSA_ERR_INVALID_ARG;
  }
  if (s->D != kD) {
    set_err("only head dim 128 is supported");
    return MSA_ERR_UNSUPPORTED;
  }
  if (s->S % kBlock != 0 || s->S > (1 << 23)) {
    set_err("S must be a multiple of 128 and at most 2^23");
    return MSA_ERR_UNSUPPORTED;
  }
  if (s->Hq % s->Hkv != 0 || s->Hq % s->Hp != 0 || (s->Hp % s->Hkv != 0 && s->Hkv % s->Hp != 0)) {
    set_err("proxy heads: Hq must be a multiple of Hkv and of Hp, and one of Hp, Hkv a multiple "
            "of the other");
    return MSA_ERR_UNSUPPORTED;
  }
  // heads per attention group: the query heads that share one selection row and one KV head
  // (the warmup forward has no selection: its groups are the GQA groups)
  const int G = op == MSA_OP_WARMUP_FORWARD ? s->Hq / s->Hkv : s->Hq / (s->Hp > s->Hkv ? s->Hp : s->Hkv);
  const bool bwd = op == MSA_OP_BACKWARD || op == MSA_OP_WARMUP_BACKWARD;
  if (!(G == 1 || G == 2 || G == 4 || G == 8 || G == 16) || (bwd && G < 4)) {
    set_err("heads per attention group, Hq / max(Hp, Hkv), must be 4, 8 or 16 (1 and 2 also "
            "allowed in the forward ops)");
    return MSA_ERR_UNSUPPORTED;
  }
  const bool sparse = op == MSA_OP_FORWARD || op == MSA_OP_BACKWARD || op == MSA_OP_DECODE;
  if (op == MSA_OP_DECODE && s->Hp > 32) {
    set_err("the decode step supports at most 32 proxy heads");
    return MSA_ERR_UNSUPPORTED;
  }
  if (sparse && (s->top_k < 1 || s->top_k > 64)) {
    set_err("top_k must be in [1, 64]");
    return MSA_ERR_UNSUPPORTED;
  }
  const long long rows = (long long)s->B * s->S * s->Hq;
  if (rows >= (1ll << 31)) {  // query rows are addressed with 32-bit TMA coordinates
    set_err("B*S*Hq must stay below 2^31");
    return MSA_ERR_UNSUPPORTED;
  }
  if (rows * kD * (sparse ? s->top_k : 1) >= (1ll << 62)) {
    set_err("problem too large");
    return MSA_ERR_UNSUPPORTED;
  }
  if ((long long)s->B * s->Hp * s->S * (sparse ? s->top_k : 1) >= (1ll << 31)) {
    set_err("B*Hp*S*top_k must stay below 2^31");
    return MSA_ERR_UNSUPPORTED;
  }
  Dims d;
  d.B = s->B;
  d.S = s->S;
  d.Hq = s->Hq;
  d.Hkv = s->Hkv;
  d.Hp = s->Hp;
  d.G = G;
  d.R = op == MSA_OP_WARMUP_FORWARD || s->Hkv <= s->Hp ? 1 : s->Hkv / s->Hp;
  d.top_k = sparse ? s->top_k : 1;
  d.nblk = s->S / kBlock;
  d.scale = s->scale;
  d = with_chunk(d, bwd ? bwd_chunk(d, sparse) : sparse ? fwd_chunk(d) : d.S);
  if (op == MSA_OP_WARMUP_BACKWARD && dense_entries(d) >= (1ll << 31)) {
    set_err("B*Hp*S*S/256 must stay below 2^31 in the warmup backward");
    return MSA_ERR_UNSUPPORTED;
  }
  *out = d;
  return MSA_OK;
}

int check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs) {
    if (!p) {
      set_err("a required pointer is null");
      return MSA_ERR_INVALID_ARG;
    }
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) {
      set_err("every pointer must be 16-byte aligned");
      return MSA_ERR_INVALID_ARG;
    }
  }
  return MSA_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// msg names the argument: a float pointer that must be 4-byte aligned.
int check_kl(const float* ptr, const char* msg) {
  if (reinterpret_cast<uintptr_t>(ptr) % 4 != 0) {
    set_err(msg);
    return MSA_ERR_INVALID_ARG;
  }
  return MSA_OK;
}

// The KL accumulator: a double at byte 128 of the workspace's status area, zeroed on the stream.
double* kl_accumulator(void* ws, const Plan& p, cudaStream_t st) {
  double* acc = at<double>(ws, p.status + 128);
  cudaMemsetAsync(acc, 0, sizeof(double), st);
  return acc;
}

int check_ws(const Plan& p, void* ws, size_t bytes) {
  if (!ws || reinterpret_cast<uintptr_t>(ws) % kAlign != 0) {
    set_err("workspace must be non-null and 256-byte aligned");
    return MSA_ERR_INVALID_ARG;
  }
  if (bytes < p.bytes) {
    snprintf(g_err, sizeof(g_err), "workspace too small: %zu < %zu bytes", bytes, p.bytes);
    return MSA_ERR_WORKSPACE;
  }
  return MSA_OK;
}

// Inverted block map + item lists shared by the sparse forward and backward.
void build_lists(const Dims& d, const Plan& p, const int32_t* idx, void* ws, int nspecs,
                 cudaStream_t st) {
  unsigned* status = at<unsigned>(ws, p.status);
  int* seg_count = at<int>(ws, p.seg_count);
  int* seg_cursor = at<int>(ws, p.seg_cursor);
  cudaMemsetAsync(seg_count, 0, d.nlist() * sizeof(int), st);
  cudaMemsetAsync(seg_cursor, 0, d.nlist() * sizeof(int), st);
  timed("invert_count", st, [&] { launch_count(d, idx, seg_count, status, st); });
  const ItemSpec specs[2] = {p.spec0, p.spec1};
  timed("invert_scan", st, [&] {
    launch_scan(d, false, seg_count, at<int>(ws, p.seg_offset), specs, nspecs, at<int>(ws, p.io0),
                nspecs > 1 ? at<int>(ws, p.io1) : nullptr, at<int>(ws, p.totals),
                at<long long>(ws, p.scan), st);
  }, scan_kernels(d.nlist()));
  timed("invert_fill", st, [&] { launch_fill(d, idx, at<int>(ws, p.seg_offset), seg_cursor, at<int>(ws, p.entries), status, st); });
  timed("work_items", st, [&] {
    launch_items(d, false, seg_count, at<int>(ws, p.seg_offset), p.spec0, at<int>(ws, p.io0),
                 at<Item>(ws, p.items0), p.max0, status, st);
  });
  if (nspecs > 1)
    timed("work_items", st, [&] {
      launch_items(d, false, seg_count, at<int>(ws, p.seg_offset), p.spec1, at<int>(ws, p.io1),
                   at<Item>(ws, p.items1),
                   p.max1, status, st);
    });
}

void zero_grads(const Dims& d, const Plan& p, void* ws, cudaStream_t st) {
  cudaMemsetAsync(at<char>(ws, p.dq), 0, (size_t)d.B * d.S * d.Hq * kD * sizeof(float), st);
  cudaMemsetAsync(at<char>(ws, p.dk), 0, (size_t)d.B * d.S * d.Hkv * kD * sizeof(float), st);
  cudaMemsetAsync(at<char>(ws, p.dv), 0, (size_t)d.B * d.S * d.Hkv * kD * sizeof(float), st);
  cudaMemsetAsync(at<char>(ws, p.dqp), 0, (size_t)d.B * d.S * d.Hp * kD * sizeof(float), st);
  cudaMemsetAsync(at<char>(ws, p.dkp), 0, (size_t)d.B * d.S * kD * sizeof(float), st);
}

// The bf16 gradients from their fp32 accumulators: the main-attention ones (dQ, dK, dV) ...
void emit_main_grads(const Dims& d, const Plan& p, void* ws, void* dq, void* dk, void* dv,
                     cudaStream_t st) {
  timed("grad_convert", st, [&] { launch_convert(at<float>(ws, p.dq), dq, (long long)d.B * d.S * d.Hq * kD, st); });
  timed("grad_convert", st, [&] { launch_convert(at<float>(ws, p.dk), dk, (long long)d.B * d.S * d.Hkv * kD, st); });
  timed("grad_convert", st, [&] { launch_convert(at<float>(ws, p.dv), dv, (long long)d.B * d.S * d.Hkv * kD, st); });
}
// ... and the proxy ones (dQp, dKp)
void emit_proxy_grads(const Dims& d, const Plan& p, void* ws, void* dqp, void* dkp, cudaStream_t st) {
  timed("grad_convert", st, [&] { launch_convert(at<float>(ws, p.dqp), dqp, (long long)d.B * d.S * d.Hp * kD, st); });
  timed("grad_convert", st, [&] { launch_convert(at<float>(ws, p.dkp), dkp, (long long)d.B * d.S * kD, st); });
}

}  // namespace

// Sets the text msa_last_error() returns on this thread (used by entry points in other files).
void set_api_error(const char* what) { set_err(what); }

}  // namespace msa

using namespace msa;

extern "C" {

size_t msa_workspace_size(const msa_shape_t* shape, int op) {
  Dims d;
  if (op < MSA_OP_FORWARD || op > MSA_OP_DECODE) return 0;
  if (check_shape(shape, op, &d) != MSA_OK) return 0;
  return make_plan(d, op).bytes;
}

int msa_forward(const msa_shape_t* shape, const void* q, const void* k, const void* v,
                const void* qp, const void* kp, int32_t* block_idx, int indices_given, void* o,
                float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  Dims d;
  int rc = check_shape(shape, MSA_OP_FORWARD, &d);
  if (rc) return rc;
  if ((rc = check_ptrs({q, k, v, block_idx, o, lse}))) return rc;
  if (!indices_given && (rc = check_ptrs({qp, kp}))) return rc;
  const Plan p = plan_for(d, MSA_OP_FORWARD, workspace_bytes);  // chunks per pass
  if ((rc = check_ws(p, workspace, workspace_bytes))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  cudaMemsetAsync(at<char>(workspace, p.status), 0, 32 * sizeof(unsigned), st);  // status, counters, wait place
  if (!indices_given) {
    bool ok = true;
    timed("proxy_topk", st, [&] {
      ok = launch_proxy_topk(d, qp, kp, block_idx, at<unsigned>(workspace, p.status), st);
    });
    if (!ok) {
      set_err("msa_forward: could not create TMA tensor maps (cuTensorMapEncodeTiled)");
      return MSA_ERR_CUDA;
    }
  }
  build_lists(d, p, block_idx, workspace, 1, st);
  // passes over consecutive sequence chunks: the items of chunks [c0, c1) are the items
  // [io0[c0 nseg], io0[c1 nseg]) of the chunk-major list, their partials indexed from c0 chunk
  const int pc = p.pass_chunks, tp = pass_tokens(d, pc);
  const int* io0 = at<int>(workspace, p.io0);
  for (int c0 = 0; c0 < d.nchunk; c0 += pc) {
    const int c1 = c0 + pc < d.nchunk ? c0 + pc : d.nchunk;
    const int t0 = c0 * d.chunk, tn = pass_tokens(d, c1) - t0;
    // partial log-sum-exps of slots no list entry reaches stay NaN (all-ones bytes)
    cudaMemsetAsync(at<float>(workspace, p.lpart), 0xff, (size_t)d.B * tp * d.Hq * d.top_k * sizeof(float), st);
    bool fok = true;
    timed("attn_fwd", st, [&] {
      fok = launch_attn_fwd(d, q, k, v, at<int>(workspace, p.seg_offset),
                            at<int>(workspace, p.entries), at<Item>(workspace, p.items0),
                            at<int>(workspace, p.totals) + 1, p.max0,
                            c0 > 0 ? io0 + (long long)c0 * d.nseg() : nullptr,
                            c1 < d.nchunk ? io0 + (long long)c1 * d.nseg() : nullptr, t0, tp,
                            at<void>(workspace, p.opart), at<float>(workspace, p.lpart),
                            at<unsigned>(workspace, p.status), st);
    });
    if (!fok) {
      set_err("msa_forward: could not create TMA tensor maps (cuTensorMapEncodeTiled)");
      return MSA_ERR_CUDA;
    }
    timed("fwd_combine", st, [&] {
      launch_combine(d, at<void>(workspace, p.opart), at<float>(workspace, p.lpart), o, lse, t0,
                     tn, tp, st);
    });
  }
  return cuda_fail("msa_forward");
}

int msa_backward(const msa_shape_t* shape, const void* q, const void* k, const void* v,
                 const void* qp, const void* kp, const void* o, const float* lse,
                 const void* dout, const int32_t* block_idx, float kl_grad,
                 const float* kl_grad_dev, void* dq, void* dk, void* dv, void* dqp, void* dkp,
                 float* kl_out, void* workspace, size_t workspace_bytes, void* stream) {
  Dims d;
  int rc = check_shape(shape, MSA_OP_BACKWARD, &d);
  if (rc) return rc;
  if ((rc = check_ptrs({q, k, v, qp, kp, o, lse, dout, block_idx, dq, dk, dv, dqp, dkp}))) return rc;
  if (kl_out && (rc = check_kl(kl_out, "kl_out must be 4-byte aligned"))) return rc;
  if (kl_grad_dev && (rc = check_kl(kl_grad_dev, "kl_grad_dev must be 4-byte aligned"))) return rc;
  const Plan p = plan_for(d, MSA_OP_BACKWARD, workspace_bytes);  // chunks per teacher pass
  if ((rc = check_ws(p, workspace, workspace_bytes))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  cudaMemsetAsync(at<char>(workspace, p.status), 0, 32 * sizeof(unsigned), st);  // status, counters, wait place
  // beside the list building and the proxy normaliser: zeroing the gradient accumulators and
  // the row data D (both HBM-bound)
  Branch pre(st);
  zero_grads(d, p, workspace, pre.aux());
  timed("bwd_rowdot", pre.aux(), [&] {
    launch_bwd_rowdot(d, o, dout, lse, at<float2>(workspace, p.rowm), pre.aux());
  });
  build_lists(d, p, block_idx, workspace, 2, st);
  // partial normalisers of slots no list entry reaches stay NaN (all-ones bytes)
  cudaMemsetAsync(at<float>(workspace, p.lpx_part), 0xff,
                  (size_t)d.B * d.S * d.Hp * d.top_k * sizeof(float), st);
  bool lok = true;
  timed("proxy_lse", st, [&] {
    lok = launch_proxy_lse_sparse(d, qp, kp, at<int>(workspace, p.seg_offset),
                                  at<int>(workspace, p.entries), at<Item>(workspace, p.items0),
                                  at<int>(workspace, p.totals) + 1, p.max0,
                                  at<float>(workspace, p.lpx_part), at<unsigned>(workspace, p.status),
                                  st);
  });
  if (!lok) {
    set_err("msa_backward: could not create TMA tensor maps (cuTensorMapEncodeTiled)");
    return MSA_ERR_CUDA;
  }
  timed("proxy_lse_combine", st, [&] {
    launch_proxy_lse_combine(d, at<float>(workspace, p.lpx_part), at<float>(workspace, p.lse_px), st);
  });
  pre.join();
  timed("entry_meta", st, [&] {
    launch_entry_meta(d, at<int>(workspace, p.seg_count), at<int>(workspace, p.seg_offset),
                      at<int>(workspace, p.entries), at<float>(workspace, p.lse_px),
                      at<float2>(workspace, p.rowm), at<float>(workspace, p.lpxe),
                      at<float2>(workspace, p.emeta), st);
  });
  // passes over consecutive sequence chunks: attn_bwd writes the teacher rows of a pass and
  // proxy_bwd reads them (the items of chunks [c0, c1) are a contiguous slice of the list)
  bool ok = true;
  double* kl_acc = kl_out ? kl_accumulator(workspace, p, st) : nullptr;
  std::unique_ptr<Branch> post;
  const int* io1 = at<int>(workspace, p.io1);
  const int* so = at<int>(workspace, p.seg_offset);
  for (int c0 = 0; c0 < d.nchunk && ok; c0 += p.pass_chunks) {
    const int c1 = c0 + p.pass_chunks < d.nchunk ? c0 + p.pass_chunks : d.nchunk;
    const int* lo = c0 > 0 ? io1 + (long long)c0 * d.nseg() : nullptr;
    const int* hi = c1 < d.nchunk ? io1 + (long long)c1 * d.nseg() : nullptr;
    const int* elo = c0 > 0 ? so + (long long)c0 * d.nseg() : nullptr;
    if (d.R > 1)  // teacher rows accumulated over the proxy head's attention groups
      cudaMemsetAsync(at<char>(workspace, p.pbar), 0, (size_t)p.pass_ent * kBlock * 2, st);
    timed("attn_bwd", st, [&] {
      ok = launch_attn_bwd(d, false, q, k, v, dout, at<float2>(workspace, p.emeta),
                           at<int>(workspace, p.seg_offset), at<int>(workspace, p.entries),
                           at<Item>(workspace, p.items1), at<int>(workspace, p.totals) + 2, p.max1,
                           lo, hi, elo, at<float>(workspace, p.dq), at<float>(workspace, p.dk),
                           at<float>(workspace, p.dv), at<void>(workspace, p.pbar),
                           at<unsigned>(workspace, p.status), st);
    });
    if (ok && c1 == d.nchunk) {
      // dQ, dK, dV are final: their conversion runs beside the last proxy backward
      post.reset(new Branch(st));
      emit_main_grads(d, p, workspace, dq, dk, dv, post->aux());
    }
    if (ok)
      timed("proxy_bwd", st, [&] {
        ok = launch_proxy_bwd(d, false, qp, kp, at<float>(workspace, p.lpxe),
                              at<void>(workspace, p.pbar), kl_grad, kl_grad_dev,
                              at<int>(workspace, p.seg_offset),
                              at<int>(workspace, p.entries), at<Item>(workspace, p.items1),
                              at<int>(workspace, p.totals) + 2, p.max1, lo, hi, elo,
                              at<float>(workspace, p.dqp), at<float>(workspace, p.dkp), kl_acc,
                              at<unsigned>(workspace, p.status), st);
      });
  }
  if (!ok) {
    set_err("msa_backward: could not create TMA tensor maps (cuTensorMapEncodeTiled)");
    return MSA_ERR_CUDA;
  }
  if (kl_out) timed("kl_finalize", st, [&] { launch_kl_finalize(d, kl_acc, kl_out, st); });
  emit_proxy_grads(d, p, workspace, dqp, dkp, st);
  if (post) post->join();
  return cuda_fail("msa_backward");
}

int msa_warmup_forward(const msa_shape_t* shape, const void* q, const void* k, const void* v,
                       void* o, float* lse, void* workspace, size_t workspace_bytes,
                       void* stream) {
  Dims d;
  int rc = check_shape(shape, MSA_OP_WARMUP_FORWARD, &d);
  if (rc) return rc;
  if ((rc = check_ptrs({q, k, v, o, lse}))) return rc;
  const Plan p = make_plan(d, MSA_OP_WARMUP_FORWARD);
  if ((rc = check_ws(p, workspace, workspace_bytes))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  cudaMemsetAsync(at<char>(workspace, p.status), 0, 32 * sizeof(unsigned), st);  // status, counters, wait place
  bool ok = true;
  timed("dense_fwd", st, [&] {
    ok = launch_dense_fwd(d, q, k, v, o, lse, at<unsigned>(workspace, p.status), st);
  });
  if (!ok) {
    set_err("msa_warmup_forward: could not create TMA tensor maps (cuTensorMapEncodeTiled)");
    return MSA_ERR_CUDA;
  }
  return cuda_fail("msa_warmup_forward");
}

int msa_warmup_backward(const msa_shape_t* shape, const void* q, const void* k, const void* v,
                        const void* qp, const void* kp, const void* o, const float* lse,
                        const void* dout, float kl_grad, const float* kl_grad_dev, void* dq,
                        void* dk, void* dv, void* dqp, void* dkp, float* kl_out, void* workspace,
                        size_t workspace_bytes, void* stream) {
  Dims d;
  int rc = check_shape(shape, MSA_OP_WARMUP_BACKWARD, &d);
  if (rc) return rc;
  if ((rc = check_ptrs({q, k, v, qp, kp, o, lse, dout, dq, dk, dv, dqp, dkp}))) return rc;
  if (kl_out && (rc = check_kl(kl_out, "kl_out must be 4-byte aligned"))) return rc;
  if (kl_grad_dev && (rc = check_kl(kl_grad_dev, "kl_grad_dev must be 4-byte aligned"))) return rc;
  const Plan p = plan_for(d, MSA_OP_WARMUP_BACKWARD, workspace_bytes);  // lists per teacher pass
  if ((rc = check_ws(p, workspace, workspace_bytes))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  unsigned* status = at<unsigned>(workspace, p.status);
  cudaMemsetAsync(status, 0, 32 * sizeof(unsigned), st);  // status, counters, wait place
  Branch pre(st);  // as in msa_backward
  zero_grads(d, p, workspace, pre.aux());
  timed("bwd_rowdot", pre.aux(), [&] {
    launch_bwd_rowdot(d, o, dout, lse, at<float2>(workspace, p.rowm), pre.aux());
  });
  const ItemSpec specs[1] = {p.spec0};
  timed("invert_scan", st, [&] {
    launch_scan(d, true, nullptr, at<int>(workspace, p.seg_offset), specs, 1,
                at<int>(workspace, p.io0), nullptr, at<int>(workspace, p.totals),
                at<long long>(workspace, p.scan), st);
  }, scan_kernels(d.nlist()));
  timed("work_items", st, [&] {
    launch_items(d, true, nullptr, at<int>(workspace, p.seg_offset), p.spec0, at<int>(workspace, p.io0),
                 at<Item>(workspace, p.items0), p.max0, status, st);
  });
  bool lok = true;
  timed("proxy_lse_dense", st, [&] {
    lok = launch_proxy_lse_dense(d, qp, kp, at<float>(workspace, p.lse_px), status, st);
  });
  if (!lok) {
    set_err("msa_warmup_backward: could not create TMA tensor maps (cuTensorMapEncodeTiled)");
    return MSA_ERR_CUDA;
  }
  pre.join();
  // passes as in msa_backward, over runs of consecutive lists [s0, s1) (the row data D and the
  // proxy normaliser are read by token, so no per-entry copy is made)
  bool ok = true;
  double* kl_acc = kl_out ? kl_accumulator(workspace, p, st) : nullptr;
  std::unique_ptr<Branch> post;
  const int* io0 = at<int>(workspace, p.io0);
  const int* so = at<int>(workspace, p.seg_offset);
  for (size_t pi = 0; pi + 1 < p.cuts.size() && ok; ++pi) {
    const long long s0 = p.cuts[pi], s1 = p.cuts[pi + 1];
    const int* lo = s0 > 0 ? io0 + s0 : nullptr;
    const int* hi = s1 < d.nlist() ? io0 + s1 : nullptr;
    const int* elo = s0 > 0 ? so + s0 : nullptr;
    if (d.R > 1)  // teacher rows accumulated over the proxy head's attention groups
      cudaMemsetAsync(at<char>(workspace, p.pbar), 0, (size_t)p.pass_ent * kBlock * 2, st);
    timed("attn_bwd_dense", st, [&] {
      ok = launch_attn_bwd(d, true, q, k, v, dout, at<float2>(workspace, p.rowm),
                           at<int>(workspace, p.seg_offset), nullptr, at<Item>(workspace, p.items0),
                           at<int>(workspace, p.totals) + 1, p.max0, lo, hi, elo,
                           at<float>(workspace, p.dq), at<float>(workspace, p.dk),
                           at<float>(workspace, p.dv), at<void>(workspace, p.pbar), status, st);
    });
    if (ok && s1 == d.nlist()) {
      post.reset(new Branch(st));
      emit_main_grads(d, p, workspace, dq, dk, dv, post->aux());
    }
    if (ok)
      timed("proxy_bwd_dense", st, [&] {
        ok = launch_proxy_bwd(d, true, qp, kp, at<float>(workspace, p.lse_px),
                              at<void>(workspace, p.pbar), kl_grad, kl_grad_dev,
                              at<int>(workspace, p.seg_offset),
                              nullptr, at<Item>(workspace, p.items0), at<int>(workspace, p.totals) + 1,
                              p.max0, lo, hi, elo, at<float>(workspace, p.dqp),
                              at<float>(workspace, p.dkp), kl_acc, status, st);
      });
  }
  if (!ok) {
    set_err("msa_warmup_backward: could not create TMA tensor maps (cuTensorMapEncodeTiled)");
    return MSA_ERR_CUDA;
  }
  if (kl_out) timed("kl_finalize", st, [&] { launch_kl_finalize(d, kl_acc, kl_out, st); });
  emit_proxy_grads(d, p, workspace, dqp, dkp, st);
  if (post) post->join();
  return cuda_fail("msa_warmup_backward");
}

int msa_decode(const msa_shape_t* shape, const void* q, const void* qp, const void* k_cache,
               const void* v_cache, const void* kp_cache, const int32_t* seq_len,
               int32_t* block_idx, void* o, float* lse, void* workspace, size_t workspace_bytes,
               void* stream) {
  Dims d;
  int rc = check_shape(shape, MSA_OP_DECODE, &d);
  if (rc) return rc;
  if ((rc = check_ptrs({q, qp, k_cache, v_cache, kp_cache, seq_len, block_idx, o, lse}))) return rc;
  const Plan p = make_plan(d, MSA_OP_DECODE);
  if ((rc = check_ws(p, workspace, workspace_bytes))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  unsigned* status = at<unsigned>(workspace, p.status);
  cudaMemsetAsync(status, 0, 32 * sizeof(unsigned), st);  // status, counters, wait place
  float* scores = at<float>(workspace, p.scores);
  bool ok = true;
  timed("decode_scores", st, [&] {
    ok = launch_decode_scores(d, qp, kp_cache, seq_len, scores, status, st);
  });
  if (!ok) {
    set_err("msa_decode: could not create TMA tensor maps (cuTensorMapEncodeTiled)");
    return MSA_ERR_CUDA;
  }
  timed("decode_select", st, [&] { launch_decode_select(d, scores, seq_len, block_idx, st); });
  timed("decode_attn", st, [&] {
    ok = launch_decode_attn(d, q, k_cache, v_cache, seq_len, block_idx, o, lse, status, st);
  });
  if (!ok) {
    set_err("msa_decode: could not create TMA tensor maps (cuTensorMapEncodeTiled)");
    return MSA_ERR_CUDA;
  }
  return cuda_fail("msa_decode");
}

int msa_device_status(void* workspace, unsigned* flags, void* stream) {
  if (!workspace || !flags) {
    set_err("workspace and flags must be non-null");
    return MSA_ERR_INVALID_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned h = 0;
  cudaGetLastError();
  cudaMemcpyAsync(&h, workspace, sizeof(unsigned), cudaMemcpyDeviceToHost, st);
  cudaMemsetAsync(workspace, 0, sizeof(unsigned), st);
  cudaStreamSynchronize(st);
  *flags = h;
  return cuda_fail("msa_device_status");
}

const char* msa_status_string(int status) {
  switch (status) {
    case MSA_OK: return "ok";
    case MSA_ERR_INVALID_ARG: return "invalid argument";
    case MSA_ERR_UNSUPPORTED: return "unsupported shape";
    case MSA_ERR_WORKSPACE: return "workspace too small";
    case MSA_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

const char* msa_last_error(void) { return g_err; }

int msa_profile_begin(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& r : g_prof) {
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_prof.clear();
  g_prof_on = true;
  return MSA_OK;
}

int msa_profile_end(char* buf, size_t len) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = false;
  std::map<std::string, std::pair<long long, double>> agg;
  std::vector<std::string> order;
  for (auto& r : g_prof) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return cuda_fail("msa_profile_end");
    float ms = 0.f;
    cudaEventElapsedTime(&ms, r.a, r.b);
    auto it = agg.find(r.name);
    if (it == agg.end()) {
      order.push_back(r.name);
      agg[r.name] = {1, ms};
    } else {
      it->second.first += 1;
      it->second.second += ms;
    }
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_prof.clear();
  std::string out;
  char line[256];
  for (auto& n : order) {
    snprintf(line, sizeof(line), "%s %lld %.6f\n", n.c_str(), agg[n].first, agg[n].second);
    out += line;
  }
  if (buf && len) {
    snprintf(buf, len, "%s", out.c_str());
  }
  return cuda_fail("msa_profile_end");
}

long long msa_launch_count(void) { return g_launches.load(); }

}  // extern "C"
