// mars_head_accept_noalloc: the LM-head + max-prob/argmax + acceptance step with its
// scratch in a fixed, library-owned device array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot call cudaMalloc at the point where they run a
// decode step — for example a serving loop whose memory is fully reserved up front and
// forbids allocation afterwards, code running inside a host framework that owns every
// device allocation and hands out no allocator, or a real-time path where an allocation
// (and the implicit synchronisation it may bring) is not allowed. They still pass the
// inputs and outputs; only the scratch moves into the library.
//
// The scratch is a file-scope __device__ array of MARS_NOALLOC_SCRATCH_BYTES. Every GPU
// that loads the library keeps that much memory reserved until the process exits. In host
// code the array's name only stands in for the symbol; its device address is looked up
// with cudaGetSymbolAddress once per device and context (on the first call made while
// that device is current) and that address is what the kernels receive.
#include <math.h>

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mars {

namespace {

// One shared scratch buffer per device (partials of the head GEMM epilogue).
static __device__ __align__(256) unsigned char g_head_scratch[MARS_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;

// The address a device's copy of g_head_scratch has in the context it was looked up in.
struct ScratchSlot {
  CUcontext ctx;
  void* ptr;
};
ScratchSlot g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry-point lookup (no link against libcuda).
CtxGetCurrentFn ctx_get_current() {
  static const CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(p);
    return static_cast<CtxGetCurrentFn>(nullptr);
  }();
  return fn;
}

// Device address of g_head_scratch on the current device. It is looked up on the first
// call made while the device is current, and again whenever the calling thread's current
// context is not the one of that lookup (after cudaDeviceReset the runtime creates a new
// primary context, in which the array has a new address).
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MARS_ECUDA;
  CUcontext ctx = nullptr;
  const CtxGetCurrentFn get = ctx_get_current();
  if (!get || get(&ctx) != CUDA_SUCCESS) return MARS_ECUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  ScratchSlot& slot = g_scratch[dev];
  if (slot.ptr == nullptr || ctx == nullptr || slot.ctx != ctx) {
    // the lookup also makes the runtime's context current when none was yet
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_head_scratch) != cudaSuccess || p == nullptr)
      return MARS_ECUDA;
    if (ctx == nullptr && (get(&ctx) != CUDA_SUCCESS || ctx == nullptr)) return MARS_ECUDA;
    slot.ctx = ctx;
    slot.ptr = p;
  }
  *out = slot.ptr;
  return MARS_OK;
}

}  // namespace

}  // namespace mars

extern "C" int mars_head_accept_noalloc(const mars_bf16* h, const mars_bf16* w, int batch,
                                        int B, int hidden, int vocab, float tau,
                                        int32_t* tokens, float* maxprob, int32_t* n_accept,
                                        int32_t* status, void* stream) {
  if (batch < 0 || B < 1 || B > 32 || hidden < 8 || vocab < 1) return MARS_EINVAL;
  if (isnan(tau) || isinf(tau)) return MARS_EINVAL;
  if (hidden % 8) return MARS_EUNSUPPORTED;
  if (batch == 0) return MARS_OK;
  if (!h || !w || !tokens || !maxprob || !n_accept) return MARS_EINVAL;
  if ((reinterpret_cast<uintptr_t>(h) & 15u) || (reinterpret_cast<uintptr_t>(w) & 15u))
    return MARS_EALIGN;
  if (mars::head_workspace_bytes(batch, B, vocab) > (size_t)MARS_NOALLOC_SCRATCH_BYTES)
    return MARS_ENOSPACE;
  void* scratch = nullptr;
  const int rc = mars::scratch_for_current_device(&scratch);
  if (rc != MARS_OK) return rc;
  // The row-block counters that must start at zero are cleared on the stream by the
  // launcher at every call; the partial records are written before they are read.
  const cudaError_t e =
      mars::launch_head_accept(h, w, batch, B, hidden, vocab, tau, nullptr, tokens, maxprob, n_accept,
                               scratch, status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MARS_OK : MARS_ECUDA;
}
