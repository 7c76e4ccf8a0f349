// Single-token decode FFN for callers that cannot allocate device memory.
//
// qffn_decode_forward needs a caller-provided workspace for the intermediate
// gate and up vectors.  Some
// callers have no way to provide one: code that runs where cudaMalloc is not
// allowed or not wanted (for example inside a host callback, in a plugin
// whose enqueue step must not allocate, or in a process whose device memory
// is entirely owned by another allocator) and that cannot keep a buffer of
// its own around between calls.  This file gives them an entry point whose
// scratch is a fixed array in the library's own device memory instead.
//
// The scratch array below lives in every GPU that loads the library, for as
// long as the process runs.  All calls on a device share it and it keeps what
// the last call wrote; the decode writes every g/u element before reading
// it, so nothing needs clearing between calls.  Calls whose execution
// overlaps on the GPU (different streams, no ordering between them) use the
// same array and race; order them on one stream or with events.
#include <cuda.h>

#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "../../include/qffn.h"
#include "launch.h"

namespace {

// Largest sizes this entry point accepts, and its scratch: g and u, H bf16 each.
constexpr int64_t kNoAllocMaxH = 32768;
constexpr int64_t kNoAllocMaxC = 32768;
constexpr size_t kScratchG = 0;
constexpr size_t kScratchU = size_t(kNoAllocMaxH) * 2;
constexpr size_t kScratchBytes = 2 * kScratchU;

static __device__ __align__(256) uint8_t g_decode_scratch[kScratchBytes];

// Device address of g_decode_scratch in each CUDA context, looked up once per
// context with it current.  In host code the array's name is only a host-side
// stand-in, never a usable device address.  The address belongs to the
// context the library's module was loaded into, so the cache is keyed on the
// current context: after cudaDeviceReset, or on a thread with another
// context current, the address is looked up again.
constexpr int kMaxContexts = 64;
std::mutex g_scratch_mu;
CUcontext g_scratch_ctx[kMaxContexts] = {nullptr};
void* g_scratch_addr[kMaxContexts] = {nullptr};
int g_scratch_n = 0;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

cudaError_t scratch_address(uint8_t** out) {
  CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  for (int i = 0; i < g_scratch_n && ctx != nullptr; ++i) {
    if (g_scratch_ctx[i] == ctx) {
      *out = static_cast<uint8_t*>(g_scratch_addr[i]);
      return cudaSuccess;
    }
  }
  // the lookup makes the current device's primary context current if no
  // context is, so the context is read again after it
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (e != cudaSuccess) return e;
  if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  // a context seen before at this slot may have been destroyed and its
  // handle reused; the newest lookup wins
  const int slot = g_scratch_n < kMaxContexts ? g_scratch_n++ : kMaxContexts - 1;
  g_scratch_ctx[slot] = ctx;
  g_scratch_addr[slot] = p;
  *out = static_cast<uint8_t*>(p);
  return cudaSuccess;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

static qffn_status decode_noalloc(uint16_t* out, const uint16_t* x,
                                  const uint8_t* w_gate, const float* s_gate,
                                  const uint8_t* w_up, const float* s_up,
                                  const uint8_t* w_down, const float* s_down,
                                  int64_t C, int64_t H, qffn_stream_t stream) {
  if (!out || !x || !w_gate || !s_gate || !w_up || !s_up || !w_down || !s_down)
    return QFFN_ERR_INVALID_ARG;
  if (C % 16 != 0 || H % 16 != 0 || C < 16 || H < 16 || C > kNoAllocMaxC || H > kNoAllocMaxH)
    return QFFN_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(out) || !aligned16(x) || !aligned16(w_gate) || !aligned16(w_up) ||
      !aligned16(w_down) || !aligned4(s_gate) || !aligned4(s_up) || !aligned4(s_down))
    return QFFN_ERR_MISALIGNED;
  uint8_t* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return QFFN_ERR_CUDA;
  uint16_t* g = reinterpret_cast<uint16_t*>(scratch + kScratchG);
  uint16_t* u = reinterpret_cast<uint16_t*>(scratch + kScratchU);
  // the same launches as qffn_decode_forward, with the scratch array as workspace
  if (qffn::launch_decode(out, x, w_gate, s_gate, w_up, s_up, w_down, s_down, C, H, g, u, false, stream) !=
      cudaSuccess)
    return QFFN_ERR_CUDA;
  return QFFN_OK;
}

extern "C" qffn_status qffn_decode_forward_noalloc(uint16_t* out, const uint16_t* x,
                                                   const uint8_t* w_gate, const float* s_gate,
                                                   const uint8_t* w_up, const float* s_up,
                                                   const uint8_t* w_down, const float* s_down,
                                                   int64_t C, int64_t H, qffn_stream_t stream) {
  nvtxRangePushA("qffn_decode_forward_noalloc");
  const qffn_status st =
      decode_noalloc(out, x, w_gate, s_gate, w_up, s_up, w_down, s_down, C, H, stream);
  nvtxRangePop();
  return st;
}
