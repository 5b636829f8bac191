// Allocation-free variant of the top-k entry point.
//
// Some callers own only their input and output buffers and cannot obtain
// device memory for a workspace: code embedded in a host framework whose
// allocator owns all device memory, or a latency-critical path that must not
// call cudaMalloc (it can synchronise the device).  hsa_topk_noalloc runs the
// same radix-select kernels as hsa_topk, with their scratch in a fixed
// file-scope device array instead of a caller workspace, and allocates
// nothing.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace hsa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device

// Zero at module load; every GPU that loads the library holds it until exit.
static __device__ __align__(256) unsigned char g_topk_scratch[kNoAllocScratchBytes];

std::mutex g_mu;

// The address is cached per device together with the unique id of the CUDA
// context it was taken in: after a cudaDeviceReset (or any other end of the
// primary context) the next call finds a different context id and looks the
// address up again instead of reusing a stale one.
struct Cached {
  unsigned long long ctx_id;
  void* addr;
};
Cached g_scratch[64] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the current thread's CUDA context (driver entry points looked
// up through the runtime, so the library needs no link against libcuda).
hsa_status_t current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  if (!get_current || !get_id) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) !=
            cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess)
      return set_error_detail(HSA_ERR_CUDA, "driver entry points cuCtxGetCurrent / cuCtxGetId");
    get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    get_id = reinterpret_cast<CtxGetIdFn>(f2);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, id) != CUDA_SUCCESS)
    return set_error_detail(HSA_ERR_CUDA, "no current CUDA context");
  return HSA_OK;
}

// Device address of the scratch array on the current device, looked up once
// per device and context (host code cannot use the symbol itself: it is a
// host-side stand-in, not a device address).
hsa_status_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error_detail(HSA_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return set_error_detail(HSA_ERR_UNSUPPORTED, "device index >= 64");
  // makes the device's primary context current (and creates it on first use)
  e = cudaSetDevice(dev);
  if (e != cudaSuccess) return set_error_detail(HSA_ERR_CUDA, cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long ctx = 0;
  hsa_status_t st = current_context_id(&ctx);
  if (st != HSA_OK) return st;
  if (!g_scratch[dev].addr || g_scratch[dev].ctx_id != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof msg, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
      return set_error_detail(HSA_ERR_CUDA, msg);
    }
    g_scratch[dev] = Cached{ctx, p};
  }
  *out = g_scratch[dev].addr;
  return HSA_OK;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace hsa

using namespace hsa;

extern "C" hsa_status_t hsa_topk_noalloc(const float* scores, const int64_t* offsets, int64_t B,
                                         int64_t total_rows, int64_t k, int32_t* idx,
                                         float* vals, void* stream) {
  if (B < 1 || B > (1 << 24)) return set_error_detail(HSA_ERR_INVALID_ARG, "B out of range");
  if (total_rows < 0 || total_rows >= (int64_t(1) << 31))
    return set_error_detail(HSA_ERR_INVALID_ARG, "total_rows out of range");
  if (k < 1) return set_error_detail(HSA_ERR_INVALID_ARG, "k must be >= 1");
  if (k > 2048) return set_error_detail(HSA_ERR_UNSUPPORTED, "k above 2048");
  if (!offsets || !idx || (!scores && total_rows > 0))
    return set_error_detail(HSA_ERR_INVALID_ARG, "null pointer");
  if (!aligned_to(offsets, 8) || !aligned_to(scores, 4) || !aligned_to(idx, 4) ||
      !aligned_to(vals, 4))
    return set_error_detail(HSA_ERR_INVALID_ARG, "misaligned pointer");
  const size_t need = topk_workspace_bytes(B, total_rows, k);
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "hsa_topk_noalloc: B=%lld, total_rows=%lld, k=%lld need %zu bytes of scratch; "
             "the static array holds %zu (use hsa_topk with a workspace)",
             (long long)B, (long long)total_rows, (long long)k, need, kNoAllocScratchBytes);
    return set_error_detail(HSA_ERR_UNSUPPORTED, msg);
  }
  void* ws = nullptr;
  hsa_status_t st = scratch_address(&ws);
  if (st != HSA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents and the layout depends on
  // (B, total_rows, k): clear the part the kernels require to start at zero.
  cudaError_t e = cudaMemsetAsync(ws, 0, topk_zero_prefix_bytes(B, total_rows, k), s);
  if (e == cudaSuccess) {
    Spans sp{offsets, nullptr, 0, 1, total_rows};
    e = launch_topk(scores, sp, static_cast<int>(B), total_rows, static_cast<int>(k), idx, vals,
                    ws, static_cast<uint32_t*>(ws), s);
  }
  if (e != cudaSuccess) return set_error_detail(HSA_ERR_CUDA, cudaGetErrorString(e));
  return HSA_OK;
}
