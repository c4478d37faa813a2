// msa_forward_noalloc: the sparse forward with its scratch in a fixed device array.
//
// For callers that cannot allocate device memory at the point of the call -- for instance code
// running inside a framework whose allocator is not reachable from its C layer, or a runtime that
// forbids allocation while it replays a recorded sequence of launches -- this entry point uses a
// file-scope __device__ array as the workspace instead of a caller-provided buffer.  Inputs and
// outputs are still the caller's.  The array is kMaxScratch bytes; every GPU that loads the
// library holds it until the process exits.
#include <stdio.h>

#include <mutex>

#include "../../include/msa.h"
#include "kernels.h"

namespace msa {
namespace {

constexpr size_t kMaxScratch = 64ull << 20;  // 64 MiB
__device__ __align__(256) unsigned char g_scratch[kMaxScratch];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};  // device address of g_scratch, per device

// Device address of the scratch array on the current device (looked up once per device; the
// name g_scratch is only a host-side stand-in and must never be passed to a kernel).
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MSA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return MSA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MSA_OK;
}

}  // namespace
}  // namespace msa

extern "C" {

int msa_forward_noalloc(const msa_shape_t* shape, const void* q, const void* k, const void* v,
                        const void* qp, const void* kp, int32_t* block_idx, int indices_given,
                        void* o, float* lse, void* stream) {
  const size_t need = msa_workspace_size(shape, MSA_OP_FORWARD);
  if (need == 0) return msa_forward(shape, q, k, v, qp, kp, block_idx, indices_given, o, lse,
                                    nullptr, 0, stream);  // reports the shape error
  if (need > msa::kMaxScratch) {
    char msg[160];
    snprintf(msg, sizeof(msg),
             "msa_forward_noalloc: shape needs %zu bytes of scratch, the fixed array holds %zu",
             need, msa::kMaxScratch);
    msa::set_api_error(msg);
    return MSA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const int rc = msa::scratch_for_current_device(&scratch);
  if (rc != MSA_OK) {
    msa::set_api_error("msa_forward_noalloc: cudaGetSymbolAddress of the scratch array failed");
    return rc;
  }
  return msa_forward(shape, q, k, v, qp, kp, block_idx, indices_given, o, lse, scratch,
                     msa::kMaxScratch, stream);
}

int msa_forward_noalloc_status(unsigned* flags, void* stream) {
  if (!flags) {
    msa::set_api_error("msa_forward_noalloc_status: flags must be non-null");
    return MSA_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  const int rc = msa::scratch_for_current_device(&scratch);
  if (rc != MSA_OK) {
    msa::set_api_error("msa_forward_noalloc_status: cudaGetSymbolAddress of the scratch array failed");
    return rc;
  }
  // the status word is the first word of the array, as of any workspace
  return msa_device_status(scratch, flags, stream);
}

}  // extern "C"
