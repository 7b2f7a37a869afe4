// mxfp8_linear_noalloc: the decode MXFP8 linear without a caller workspace.
//
// Some callers cannot call cudaMalloc or hand the library a scratch buffer:
// engines that plan every byte of device memory before serving and forbid
// allocation on the request path (an allocation there can stall, fragment the
// pool or fail with out-of-memory at an unpredictable moment), and plugin or
// callback code that a host framework gives only its input and output tensors
// while the framework keeps the device allocator to itself.  This entry point
// serves them: it runs the same quantizer + split-K GEMV launches as
// mxfp8_linear's workspace path, with the scratch (the quantized activation and
// its codes) in a fixed library-owned device array instead of caller memory.
//
// The array is a file-scope __device__ variable of MX_NOALLOC_SCRATCH_BYTES;
// every GPU that loads the library holds one until the process exits.  Host
// code must not pass the array's name to a kernel (on the host it is only a
// stand-in, not a device address): the device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, on the first
// call made on it.  The address belongs to the device's context: when that
// context is replaced (cudaDeviceReset, or the primary context released and
// created again) the module is loaded anew, so the lookup is keyed by the
// context's unique id and made again for a new context.  All calls share the
// array and each call overwrites what the previous one left there; every byte
// a call reads it writes first, so nothing needs clearing.

#include <cudaTypedefs.h>

#include <mutex>

#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[MX_NOALLOC_SCRATCH_BYTES];

struct ScratchSlot {
  void* ptr;                   // device address of the array in that context
  unsigned long long ctx_id;   // unique id of the context it was looked up in
};
std::mutex g_scratch_mu;
ScratchSlot g_scratch[64] = {};

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

// Unique id of the context current on this thread; false when there is none
// yet (or the driver cannot say), in which case the address is looked up again.
bool current_context_id(unsigned long long* id) {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  if (!g_ctx_current || !g_ctx_id) return false;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the current device's scratch array: looked up with
// cudaGetSymbolAddress (that device current) on the first call in a context,
// then taken from the cache while the context stays the same.
int scratch_for_current_device(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return set_error(MX_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  if (!have_id || g_scratch[dev].ptr == nullptr || g_scratch[dev].ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return set_error(MX_ERR_CUDA, "cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
    // the lookup made the device's context current if it was not yet
    unsigned long long id_now = 0;
    g_scratch[dev].ptr = p;
    g_scratch[dev].ctx_id = current_context_id(&id_now) ? id_now : 0ull;
    *out = static_cast<uint8_t*>(p);
    return MX_OK;
  }
  *out = static_cast<uint8_t*>(g_scratch[dev].ptr);
  return MX_OK;
}

}  // namespace
}  // namespace mx

using namespace mx;

extern "C" int mxfp8_linear_noalloc(const void* x, int M, const mx_packed_weight* w, const void* bias,
                                    void* out, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!w) return set_error(MX_ERR_ARG, "NULL weight");
  if (w->fmt != MX_FMT_E4M3 || w->E != 1)
    return set_error(MX_ERR_ARG, "mxfp8_linear_noalloc needs a dense E4M3 weight");
  if (M < 0) return set_error(MX_ERR_SHAPE, "M=%d", M);
  if (M == 0) return MX_OK;
  if (M > MX_GEMV_MAX_M)
    return set_error(MX_ERR_UNSUPPORTED, "mxfp8_linear_noalloc serves at most %d tokens, got M=%d",
                     MX_GEMV_MAX_M, M);
  if (!x || !out) return set_error(MX_ERR_ARG, "NULL pointer");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out) |
       reinterpret_cast<uintptr_t>(bias)) & 15u)
    return set_error(MX_ERR_ALIGN, "x, out and bias need 16-byte alignment");
  // scratch: quantized activation [M, Kp] then its codes [M, Kp/32]
  const size_t Kp = static_cast<size_t>(w->Kp);
  const size_t codes_off = (static_cast<size_t>(M) * Kp + 255) / 256 * 256;
  const size_t need = codes_off + static_cast<size_t>(M) * (Kp / 32);
  if (need > MX_NOALLOC_SCRATCH_BYTES)
    return set_error(MX_ERR_UNSUPPORTED,
                     "M=%d, K=%d needs %zu bytes of scratch; the fixed scratch array holds %u", M, w->K,
                     need, static_cast<unsigned>(MX_NOALLOC_SCRATCH_BYTES));
  DeviceInfo di;
  int rc = current_device_info(&di);
  if (rc != MX_OK) return rc;
  if (di.cc_major != 10 || di.cc_minor != 3)
    return set_error(MX_ERR_UNSUPPORTED, "device compute capability %d.%d is not sm_103", di.cc_major,
                     di.cc_minor);
  uint8_t* scratch = nullptr;
  if ((rc = scratch_for_current_device(&scratch)) != MX_OK) return rc;
  uint8_t* xq = scratch;
  uint8_t* xcodes = scratch + codes_off;
  cudaError_t e = launch_quant_act(x, M, w->K, w->Kp, xq, w->Kp, xcodes, w->Kp / 32, 127, nullptr, true, stream);
  if (e != cudaSuccess) return set_error(MX_ERR_CUDA, "quantize launch: %s", cudaGetErrorString(e));
  GemvArgs a = {};
  a.w = w;
  a.x = x;
  a.xq = xq;
  a.xcodes = xcodes;
  a.bias = bias;
  a.out = out;
  a.M = M;
  a.fused = false;
  a.pdl = true;
  return launch_gemv(a, stream);
}
