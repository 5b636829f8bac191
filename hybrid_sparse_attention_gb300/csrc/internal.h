// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hsa.h"

#if defined(__CUDACC__)
#define HSA_HOST_DEVICE __host__ __device__ inline
#else
#define HSA_HOST_DEVICE inline
#endif

namespace hsa {

struct Spans;

// Records `detail` as this thread's hsa_last_error_detail() text; returns s.
hsa_status_t set_error_detail(hsa_status_t s, const char* detail);

// Streaming multiprocessors of the current device (cached per device).
int device_sms();

// The bound on a kernel's pipeline waits (hsa_set_wait_limit; process-wide):
// nanoseconds and polls after which a wait gives up with HSA_DEV_TIMEOUT.
uint64_t wait_limit_ns();
uint32_t wait_limit_polls();

// Kernel launch; with pdl, the kernel may be scheduled while the previous
// kernel of the stream is still running (it waits for it in pdl_wait).  With
// cluster > 0, consecutive groups of `cluster` CTAs (along x) form thread-block
// clusters (for kernels without a compile-time cluster shape).
template <typename... KArgs, typename... Args>
cudaError_t launch_kc(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t stream, bool pdl, unsigned cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t stream, bool pdl, Args... args) {
  return launch_kc(kernel, grid, block, smem, stream, pdl, 0u, args...);
}

// overlap: the C4 overlap transform (entry n over blocks n-1 and n, b [2r, C]).
cudaError_t launch_compress(const void* kv, const void* z, const float* b, int64_t S, int64_t T,
                            int64_t C, int64_t r, void* out, int out_dtype, cudaStream_t stream,
                            bool overlap = false);

// 2-D bf16 tensor map (inner dimension contiguous) for TMA tiled loads.
cudaError_t make_tmap_2d_bf16(CUtensorMap* map, const void* base, int64_t inner, int64_t outer,
                              int box_inner, int box_outer, CUtensorMapSwizzle swizzle);
// The same over bytes (8-bit elements, e.g. E4M3 codes).
cudaError_t make_tmap_2d_u8(CUtensorMap* map, const void* base, int64_t inner, int64_t outer,
                            int box_inner, int box_outer, CUtensorMapSwizzle swizzle);

// Per-row E4M3 quantization of an fp32 [rows, C] matrix (C a multiple of 4):
// scale = amax / 448, code = e4m3(x * (448 / amax)), rounded to nearest even
// and saturated; a zero row gets scale 0 and zero codes.
cudaError_t launch_quantize_e4m3(const float* x, int64_t rows, int64_t C, uint8_t* codes,
                                 float* scales, cudaStream_t stream);

size_t indexer_smem_bytes(int Di, bool fp8 = false);
// With pdl, wait_mode says where the kernel waits for the previous one: 0
// every thread at the start; 1 the loads (the tile table is built before,
// from sp, which the previous kernel must not write); 2 only the loads of a
// tile holding a row the previous kernel may have written (the last live row
// of a sequence whose length, per sp, completes a block), the next kernel
// being triggered first (it must read nothing the previous kernel writes
// before its own wait).
// row_hist (may be null): B x kRowHistBins counters to which every score
// written adds one in the bin of its top kRowHistBits order-key bits.
// key_scale non-null: keys are E4M3 codes [total_rows, Di] (Di = 128) with one
// fp32 scale per row, and the kernel quantizes each (sequence, head) query
// row of iq the same way (E4M3 tensor-core products, fp32 accumulation).
// T query tokens per sequence (T * Hi <= 16): iq [B, T, Hi, Di], w [B, T, Hi];
// sp counts the sequence's rows for its last token; token t scores the rows
// visible to it into scores + t * total_rows (row_hist: B * T histograms).
cudaError_t launch_indexer(const void* iq, const float* w, const void* keys, Spans sp, int B, int Hi,
                           int Di, int64_t total_rows, float* scores, uint32_t* status,
                           cudaStream_t stream, bool pdl = false, int wait_mode = 0,
                           uint32_t* row_hist = nullptr, const float* key_scale = nullptr,
                           int T = 1);

size_t topk_workspace_bytes(int64_t B, int64_t total_rows, int64_t k);
// Leading bytes of a top-k workspace (status word, row states, histograms)
// that must be zero when a call starts.
size_t topk_zero_prefix_bytes(int64_t B, int64_t total_rows, int64_t k);
// max_row: a bound on every row's length (0 = unknown).  When it (or
// total_rows) is at most 32768, one clustered launch handles every row and a
// longer row is flagged as out of bounds and treated as empty.
cudaError_t launch_topk(const float* scores, Spans sp, int B, int64_t total_rows, int k,
                        int32_t* idx, float* vals, void* ws, uint32_t* status,
                        cudaStream_t stream, int64_t max_row = 0, bool pdl = false);

// The top-k workspace's candidate area (one 8-byte slot per score).
uint64_t* topk_cand_area(void* ws, int64_t B, int64_t total_rows, int64_t k);

size_t layer_workspace_bytes(const hsa_layer_desc& d);
int layer_launch_count(const hsa_layer_desc& d);
// Kernel launches launch_topk makes for these arguments.
int topk_launch_count(int64_t total_rows, int64_t max_row);
cudaError_t launch_layer(const hsa_layer_desc& d, void* ws, cudaStream_t stream);

}  // namespace hsa
