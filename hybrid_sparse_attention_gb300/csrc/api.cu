// C ABI: host-side validation, status handling and kernel launches.
//
// Nothing here computes: every step of the path runs in the kernels of this
// library.  Each entry point validates its arguments before any launch and
// returns an hsa_status_t; no C++ exception crosses the boundary.
#include <cstdarg>
#include <cstdio>
#include <cmath>
#include <cstring>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace hsa {
namespace {

thread_local char g_detail[512] = "";

hsa_status_t fail(hsa_status_t s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof g_detail, fmt, ap);
  va_end(ap);
  return s;
}

hsa_status_t cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return HSA_OK;
  return fail(HSA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

hsa_status_t set_error_detail(hsa_status_t s, const char* detail) {
  snprintf(g_detail, sizeof g_detail, "%s", detail);
  return s;
}

int device_sms() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

namespace {

cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType type, int esize,
                         int64_t inner, int64_t outer, int box_inner, int box_outer,
                         CUtensorMapSwizzle swizzle) {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                       cudaEnableDefault, &q);
      if (e != cudaSuccess) return e;
      if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * esize};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

namespace {
constexpr uint64_t kDefaultWaitNs = 200ull * 1000 * 1000;  // 200 ms
constexpr uint32_t kDefaultWaitPolls = 1u << 24;
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<uint32_t> g_wait_polls{kDefaultWaitPolls};
}  // namespace

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
uint32_t wait_limit_polls() { return g_wait_polls.load(std::memory_order_relaxed); }

cudaError_t make_tmap_2d_bf16(CUtensorMap* map, const void* base, int64_t inner, int64_t outer,
                              int box_inner, int box_outer, CUtensorMapSwizzle swizzle) {
  return make_tmap_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, outer, box_inner,
                      box_outer, swizzle);
}

cudaError_t make_tmap_2d_u8(CUtensorMap* map, const void* base, int64_t inner, int64_t outer,
                            int box_inner, int box_outer, CUtensorMapSwizzle swizzle) {
  return make_tmap_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, inner, outer, box_inner,
                      box_outer, swizzle);
}

}  // namespace hsa

using namespace hsa;

#define HSA_CHECK(cond, code, ...)      \
  do {                                  \
    if (!(cond)) return fail(code, __VA_ARGS__); \
  } while (0)

extern "C" {

const char* hsa_status_string(hsa_status_t s) {
  switch (s) {
    case HSA_OK: return "HSA_OK";
    case HSA_ERR_INVALID_ARG: return "HSA_ERR_INVALID_ARG";
    case HSA_ERR_UNSUPPORTED: return "HSA_ERR_UNSUPPORTED";
    case HSA_ERR_CUDA: return "HSA_ERR_CUDA";
    case HSA_ERR_DEVICE_BOUNDS: return "HSA_ERR_DEVICE_BOUNDS";
    case HSA_ERR_TIMEOUT: return "HSA_ERR_TIMEOUT";
    case HSA_ERR_WORKSPACE: return "HSA_ERR_WORKSPACE";
    case HSA_ERR_NAN: return "HSA_ERR_NAN";
  }
  return "HSA_ERR_UNKNOWN";
}

const char* hsa_last_error_detail(void) { return g_detail; }

int hsa_version(void) { return 100; }

hsa_status_t hsa_workspace_status(void* ws, void* stream, uint32_t* bits) {
  HSA_CHECK(ws, HSA_ERR_WORKSPACE, "workspace is null");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  hsa_status_t s = cuda_status(cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, st),
                               "status read");
  if (s != HSA_OK) return s;
  s = cuda_status(cudaStreamSynchronize(st), "status sync");
  if (s != HSA_OK) return s;
  s = cuda_status(cudaMemsetAsync(ws, 0, sizeof v, st), "status clear");
  if (s != HSA_OK) return s;
  if (bits) *bits = v;
  if (v & HSA_DEV_BOUNDS) return fail(HSA_ERR_DEVICE_BOUNDS, "device saw an out-of-range index");
  if (v & HSA_DEV_TIMEOUT) return fail(HSA_ERR_TIMEOUT, "a device wait ran out");
  if (v & HSA_DEV_NAN) return fail(HSA_ERR_NAN, "NaN score reached the top-k");
  return HSA_OK;
}

static hsa_status_t compress_call(const void* kv, const void* z, const float* b, int64_t S,
                                  int64_t T, int64_t C, int64_t r, void* out, int out_dtype,
                                  void* stream, bool overlap) {
  HSA_CHECK(S >= 0 && T >= 0, HSA_ERR_INVALID_ARG, "S=%lld T=%lld must be >= 0", (long long)S,
            (long long)T);
  HSA_CHECK(C > 0 && C % 8 == 0, HSA_ERR_UNSUPPORTED, "C=%lld must be a positive multiple of 8",
            (long long)C);
  HSA_CHECK(r >= 1 && r <= (overlap ? 2048 : 4096), HSA_ERR_UNSUPPORTED, "r=%lld outside [1, %d]",
            (long long)r, overlap ? 2048 : 4096);
  HSA_CHECK(out_dtype == HSA_F32 || out_dtype == HSA_BF16, HSA_ERR_INVALID_ARG, "bad out_dtype");
  if (S == 0 || T / r == 0) return HSA_OK;
  HSA_CHECK(kv && z && b && out, HSA_ERR_INVALID_ARG, "null pointer");
  HSA_CHECK(aligned(kv, 16) && aligned(z, 16) && aligned(b, 16) && aligned(out, 16),
            HSA_ERR_INVALID_ARG, "kv, z, b and out must be 16-byte aligned");
  return cuda_status(launch_compress(kv, z, b, S, T, C, r, out, out_dtype,
                                     static_cast<cudaStream_t>(stream), overlap),
                     "compress launch");
}

hsa_status_t hsa_compress(const void* kv, const void* z, const float* b, int64_t S, int64_t T,
                          int64_t C, int64_t r, void* out, int out_dtype, void* stream) {
  return compress_call(kv, z, b, S, T, C, r, out, out_dtype, stream, false);
}

hsa_status_t hsa_compress_overlap(const void* kv, const void* z, const float* b, int64_t S,
                                  int64_t T, int64_t C, int64_t r, void* out, int out_dtype,
                                  void* stream) {
  return compress_call(kv, z, b, S, T, C, r, out, out_dtype, stream, true);
}

size_t hsa_indexer_scores_workspace_size(void) { return kWsHeader; }

hsa_status_t hsa_indexer_scores(const void* iq, const float* w, const void* keys,
                                const int64_t* offsets, int64_t B, int64_t Hi, int64_t Di,
                                int64_t total_rows, float* scores, void* ws, size_t ws_bytes,
                                void* stream) {
  HSA_CHECK(B >= 1 && B <= (1 << 24), HSA_ERR_INVALID_ARG, "B=%lld out of range", (long long)B);
  HSA_CHECK(B <= 4096, HSA_ERR_UNSUPPORTED, "B=%lld above the indexer's 4096 sequences",
            (long long)B);
  HSA_CHECK(Hi >= 1 && Hi <= 16, HSA_ERR_UNSUPPORTED, "Hi=%lld outside [1, 16]", (long long)Hi);
  HSA_CHECK(Di == 32 || Di == 64 || Di == 128, HSA_ERR_UNSUPPORTED, "Di=%lld not in {32, 64, 128}",
            (long long)Di);
  HSA_CHECK(total_rows >= 0 && total_rows < (int64_t(1) << 31), HSA_ERR_INVALID_ARG,
            "total_rows=%lld out of range", (long long)total_rows);
  HSA_CHECK(iq && w && offsets && (keys || total_rows == 0) && (scores || total_rows == 0),
            HSA_ERR_INVALID_ARG, "null pointer");
  HSA_CHECK(aligned(iq, 16) && aligned(keys, 16) && aligned(w, 4) && aligned(scores, 4) &&
                aligned(offsets, 8),
            HSA_ERR_INVALID_ARG, "misaligned pointer (iq, keys: 16 bytes)");
  HSA_CHECK(ws && aligned(ws, 256) && ws_bytes >= kWsHeader, HSA_ERR_WORKSPACE,
            "workspace null, misaligned or below %zu bytes", kWsHeader);
  Spans sp{offsets, nullptr, 0, 1, total_rows};
  return cuda_status(launch_indexer(iq, w, keys, sp, static_cast<int>(B), static_cast<int>(Hi),
                                    static_cast<int>(Di), total_rows, scores,
                                    static_cast<uint32_t*>(ws), static_cast<cudaStream_t>(stream)),
                     "indexer launch");
}

hsa_status_t hsa_set_wait_limit(uint64_t nanos, uint32_t polls) {
  g_wait_ns.store(nanos == 0 ? kDefaultWaitNs : nanos, std::memory_order_relaxed);
  g_wait_polls.store(polls == 0 ? kDefaultWaitPolls : polls, std::memory_order_relaxed);
  return HSA_OK;
}

hsa_status_t hsa_quantize_e4m3(const float* x, int64_t rows, int64_t C, uint8_t* codes,
                               float* scales, void* stream) {
  HSA_CHECK(rows >= 0 && rows < (int64_t(1) << 34), HSA_ERR_INVALID_ARG, "rows=%lld out of range",
            (long long)rows);
  HSA_CHECK(C > 0 && C % 4 == 0 && C < (int64_t(1) << 30), HSA_ERR_UNSUPPORTED,
            "C=%lld must be a positive multiple of 4", (long long)C);
  if (rows == 0) return HSA_OK;
  HSA_CHECK(x && codes && scales, HSA_ERR_INVALID_ARG, "null pointer");
  HSA_CHECK(aligned(x, 16) && aligned(codes, 4) && aligned(scales, 4), HSA_ERR_INVALID_ARG,
            "misaligned pointer (x: 16 bytes, codes: 4)");
  return cuda_status(launch_quantize_e4m3(x, rows, C, codes, scales,
                                          static_cast<cudaStream_t>(stream)),
                     "quantize launch");
}

hsa_status_t hsa_indexer_scores_e4m3(const void* iq, const float* w, const uint8_t* keys,
                                     const float* key_scales, const int64_t* offsets, int64_t B,
                                     int64_t Hi, int64_t Di, int64_t total_rows, float* scores,
                                     void* ws, size_t ws_bytes, void* stream) {
  HSA_CHECK(B >= 1 && B <= (1 << 24), HSA_ERR_INVALID_ARG, "B=%lld out of range", (long long)B);
  HSA_CHECK(B <= 4096, HSA_ERR_UNSUPPORTED, "B=%lld above the indexer's 4096 sequences",
            (long long)B);
  HSA_CHECK(Hi >= 1 && Hi <= 16, HSA_ERR_UNSUPPORTED, "Hi=%lld outside [1, 16]", (long long)Hi);
  HSA_CHECK(Di == 128, HSA_ERR_UNSUPPORTED, "Di=%lld: E4M3 keys need Di = 128", (long long)Di);
  HSA_CHECK(total_rows >= 0 && total_rows < (int64_t(1) << 31), HSA_ERR_INVALID_ARG,
            "total_rows=%lld out of range", (long long)total_rows);
  HSA_CHECK(iq && w && offsets && (keys || total_rows == 0) && (key_scales || total_rows == 0) &&
                (scores || total_rows == 0),
            HSA_ERR_INVALID_ARG, "null pointer");
  HSA_CHECK(aligned(iq, 16) && aligned(keys, 16) && aligned(w, 4) && aligned(scores, 4) &&
                aligned(key_scales, 4) && aligned(offsets, 8),
            HSA_ERR_INVALID_ARG, "misaligned pointer (iq, keys: 16 bytes)");
  HSA_CHECK(ws && aligned(ws, 256) && ws_bytes >= kWsHeader, HSA_ERR_WORKSPACE,
            "workspace null, misaligned or below %zu bytes", kWsHeader);
  Spans sp{offsets, nullptr, 0, 1, total_rows};
  return cuda_status(launch_indexer(iq, w, keys, sp, static_cast<int>(B), static_cast<int>(Hi),
                                    static_cast<int>(Di), total_rows, scores,
                                    static_cast<uint32_t*>(ws), static_cast<cudaStream_t>(stream),
                                    false, 0, nullptr, key_scales),
                     "indexer launch");
}

size_t hsa_decode_attn_workspace_size(int64_t B, int64_t Hq, int64_t Dqk, int64_t Dv, int64_t W,
                                      int64_t extra_slots) {
  if (B < 1 || Hq < 1 || Dqk < 1 || Dv < 1 || W < 0 || extra_slots < 0) return 0;
  return attn_workspace_bytes(attn_plan(B, Hq, Dqk, Dv, W, extra_slots), B, Hq, Dv);
}

static hsa_status_t check_attn_shape(int64_t B, int64_t Hq, int64_t Dqk, int64_t Dv, int64_t W) {
  HSA_CHECK(B >= 1 && B <= (1 << 20), HSA_ERR_INVALID_ARG, "B=%lld out of range", (long long)B);
  HSA_CHECK(W >= 0 && W <= (1 << 24), HSA_ERR_INVALID_ARG, "W=%lld out of range", (long long)W);
  HSA_CHECK(Hq >= 1 && (Hq <= 32 || Hq % 32 == 0) && Hq <= 1024, HSA_ERR_UNSUPPORTED,
            "Hq=%lld: need Hq <= 32 or a multiple of 32", (long long)Hq);
  HSA_CHECK(Dqk % 64 == 0 && Dqk >= 128 && Dqk <= 576, HSA_ERR_UNSUPPORTED,
            "Dqk=%lld: need a multiple of 64 in [128, 576]", (long long)Dqk);
  HSA_CHECK(Dv % 128 == 0 && Dv >= 128 && Dv <= Dqk, HSA_ERR_UNSUPPORTED,
            "Dv=%lld: need a multiple of 128 in [128, Dqk]", (long long)Dv);
  return HSA_OK;
}

hsa_status_t hsa_decode_attn(const void* q, const void* swa, const int32_t* seq_len, int64_t W,
                             const void* extra, const int64_t* extra_offsets,
                             int64_t extra_total_rows, const int32_t* extra_idx, int64_t k,
                             int64_t max_extra_rows, int64_t B, int64_t Hq, int64_t Dqk,
                             int64_t Dv, float scale, void* out, int out_dtype, float* lse,
                             void* ws, size_t ws_bytes, void* stream) {
  hsa_status_t st = check_attn_shape(B, Hq, Dqk, Dv, W);
  if (st != HSA_OK) return st;
  HSA_CHECK(q && seq_len && out && (swa || W == 0), HSA_ERR_INVALID_ARG, "null pointer");
  HSA_CHECK(out_dtype == HSA_F32 || out_dtype == HSA_BF16, HSA_ERR_INVALID_ARG, "bad out_dtype");
  HSA_CHECK(isfinite(scale), HSA_ERR_INVALID_ARG, "scale must be finite");
  HSA_CHECK(aligned(q, 16) && aligned(swa, 16) && aligned(extra, 16) && aligned(out, 16) &&
                aligned(lse, 4) && aligned(seq_len, 4) && aligned(extra_offsets, 8) &&
                aligned(extra_idx, 4),
            HSA_ERR_INVALID_ARG, "misaligned pointer (q, swa, extra, out: 16 bytes)");
  int64_t slots = 0;
  if (extra) {
    HSA_CHECK(extra_offsets, HSA_ERR_INVALID_ARG, "extra given without extra_offsets");
    HSA_CHECK(extra_total_rows >= 0, HSA_ERR_INVALID_ARG, "extra_total_rows < 0");
    if (extra_idx) {
      HSA_CHECK(k >= 1 && k <= (1 << 16), HSA_ERR_INVALID_ARG, "k=%lld out of range", (long long)k);
      slots = k;
    } else {
      HSA_CHECK(max_extra_rows >= 0 && max_extra_rows <= (int64_t(1) << 28), HSA_ERR_INVALID_ARG,
                "max_extra_rows=%lld out of range", (long long)max_extra_rows);
      slots = max_extra_rows;
    }
  } else {
    HSA_CHECK(!extra_idx, HSA_ERR_INVALID_ARG, "extra_idx given without extra");
  }
  const AttnPlan pl = attn_plan(B, Hq, Dqk, Dv, W, slots);
  const size_t need = attn_workspace_bytes(pl, B, Hq, Dv);
  HSA_CHECK(ws && aligned(ws, 256) && ws_bytes >= need, HSA_ERR_WORKSPACE,
            "workspace null, misaligned or below %zu bytes", need);
  AttnArgs a;
  a.q = q;
  a.swa = swa;
  a.seq_len = seq_len;
  a.len_add = 0;
  a.W = W;
  a.extra = extra;
  a.sp = Spans{extra_offsets, nullptr, 0, 1, extra_total_rows};
  a.idx = extra ? extra_idx : nullptr;
  a.k = extra_idx ? k : 0;
  a.max_rows = extra_idx ? 0 : max_extra_rows;
  a.B = B;
  a.Hq = Hq;
  a.Dqk = Dqk;
  a.Dv = Dv;
  a.scale = scale;
  a.out = out;
  a.out_dtype = out_dtype;
  a.lse = lse;
  return cuda_status(launch_attn(a, pl, ws, static_cast<uint32_t*>(ws),
                                 static_cast<cudaStream_t>(stream)),
                     "attention launch");
}

static hsa_status_t check_layer(const hsa_layer_desc* d) {
  HSA_CHECK(d, HSA_ERR_INVALID_ARG, "null descriptor");
  HSA_CHECK(d->kind == HSA_LAYER_C4 || d->kind == HSA_LAYER_C128, HSA_ERR_INVALID_ARG,
            "kind=%d not HSA_LAYER_C4 / HSA_LAYER_C128", d->kind);
  hsa_status_t st = check_attn_shape(d->B, d->Hq, d->Dqk, d->Dv, d->W);
  if (st != HSA_OK) return st;
  HSA_CHECK(d->W >= 1, HSA_ERR_INVALID_ARG, "W must be >= 1");
  HSA_CHECK(d->out_dtype == HSA_F32 || d->out_dtype == HSA_BF16, HSA_ERR_INVALID_ARG,
            "bad out_dtype");
  HSA_CHECK(isfinite(d->scale), HSA_ERR_INVALID_ARG, "scale must be finite");
  HSA_CHECK(d->pool_total_rows >= 0 && d->pool_total_rows < (int64_t(1) << 31),
            HSA_ERR_INVALID_ARG, "pool_total_rows out of range");
  HSA_CHECK(d->seq_len_in && d->seq_len_out && d->pool_offsets && d->kv_new && d->z_new &&
                d->b_kv && d->swa && d->kv_ring && d->z_ring && d->kv_pool && d->q && d->out,
            HSA_ERR_INVALID_ARG, "null pointer in descriptor");
  HSA_CHECK(aligned(d->kv_new, 16) && aligned(d->z_new, 16) && aligned(d->b_kv, 16) &&
                aligned(d->swa, 16) && aligned(d->kv_ring, 16) && aligned(d->z_ring, 16) &&
                aligned(d->kv_pool, 16) && aligned(d->q, 16) && aligned(d->out, 16) &&
                aligned(d->pool_offsets, 8) && aligned(d->lse, 4),
            HSA_ERR_INVALID_ARG, "misaligned pointer in descriptor");
  HSA_CHECK(d->T >= 0 && d->T <= 4, HSA_ERR_UNSUPPORTED, "T=%d outside [0, 4]", d->T);
  if (d->kind == HSA_LAYER_C4) {
    HSA_CHECK(d->B <= 4096, HSA_ERR_UNSUPPORTED, "B=%d above the indexer's 4096 sequences", d->B);
    HSA_CHECK(d->Hi * (d->T > 1 ? d->T : 1) <= 16, HSA_ERR_UNSUPPORTED,
              "T * Hi = %d above the indexer's 16 query rows", d->Hi * (d->T > 1 ? d->T : 1));
    HSA_CHECK(d->Hi >= 1 && d->Hi <= 16, HSA_ERR_UNSUPPORTED, "Hi=%d outside [1, 16]", d->Hi);
    HSA_CHECK(d->Di == 32 || d->Di == 64 || d->Di == 128, HSA_ERR_UNSUPPORTED,
              "Di=%d not in {32, 64, 128}", d->Di);
    HSA_CHECK(d->k >= 1 && d->k <= 2048, HSA_ERR_UNSUPPORTED, "k=%d outside [1, 2048]", d->k);
    HSA_CHECK(d->ik_new && d->iz_new && d->b_ik && d->ik_ring && d->iz_ring && d->key_pool &&
                  d->iq && d->w,
              HSA_ERR_INVALID_ARG, "C4 layer needs the indexer tensors");
    HSA_CHECK(aligned(d->ik_new, 16) && aligned(d->iz_new, 16) && aligned(d->b_ik, 16) &&
                  aligned(d->ik_ring, 16) && aligned(d->iz_ring, 16) &&
                  aligned(d->key_pool, 16) && aligned(d->iq, 16) && aligned(d->w, 4) &&
                  aligned(d->topk_idx, 4) && aligned(d->scores, 4),
              HSA_ERR_INVALID_ARG, "misaligned indexer pointer");
    HSA_CHECK(d->key_fp8 == 0 || d->key_fp8 == 1, HSA_ERR_INVALID_ARG, "key_fp8 must be 0 or 1");
    if (d->key_fp8) {
      HSA_CHECK(d->Di == 128, HSA_ERR_UNSUPPORTED, "Di=%d: E4M3 keys need Di = 128", d->Di);
      HSA_CHECK(d->key_scale && aligned(d->key_scale, 4), HSA_ERR_INVALID_ARG,
                "E4M3 keys need an aligned key_scale");
    }
  } else {
    HSA_CHECK(d->max_pool_rows >= 0 && d->max_pool_rows <= (int64_t(1) << 28),
              HSA_ERR_INVALID_ARG, "max_pool_rows out of range");
  }
  return HSA_OK;
}

size_t hsa_layer_decode_workspace_size(const hsa_layer_desc* d) {
  if (check_layer(d) != HSA_OK) return 0;
  return layer_workspace_bytes(*d);
}

int32_t hsa_layer_decode_launches(const hsa_layer_desc* d) {
  if (check_layer(d) != HSA_OK) return 0;
  return layer_launch_count(*d);
}

hsa_status_t hsa_layer_decode(const hsa_layer_desc* d, void* ws, size_t ws_bytes, void* stream) {
  hsa_status_t st = check_layer(d);
  if (st != HSA_OK) return st;
  const size_t need = layer_workspace_bytes(*d);
  HSA_CHECK(ws && aligned(ws, 256) && ws_bytes >= need, HSA_ERR_WORKSPACE,
            "workspace null, misaligned or below %zu bytes", need);
  return cuda_status(launch_layer(*d, ws, static_cast<cudaStream_t>(stream)), "layer launch");
}

size_t hsa_topk_workspace_size(int64_t B, int64_t total_rows, int64_t k) {
  if (B < 1 || total_rows < 0 || k < 1) return 0;
  return topk_workspace_bytes(B, total_rows, k);
}

hsa_status_t hsa_topk(const float* scores, const int64_t* offsets, int64_t B, int64_t total_rows,
                      int64_t k, int32_t* idx, float* vals, void* ws, size_t ws_bytes,
                      void* stream) {
  HSA_CHECK(B >= 1 && B <= (1 << 24), HSA_ERR_INVALID_ARG, "B=%lld out of range", (long long)B);
  HSA_CHECK(total_rows >= 0 && total_rows < (int64_t(1) << 31), HSA_ERR_INVALID_ARG,
            "total_rows=%lld out of range", (long long)total_rows);
  HSA_CHECK(k >= 1, HSA_ERR_INVALID_ARG, "k=%lld must be >= 1", (long long)k);
  HSA_CHECK(k <= 2048, HSA_ERR_UNSUPPORTED, "k=%lld above 2048", (long long)k);
  HSA_CHECK(offsets && idx, HSA_ERR_INVALID_ARG, "null pointer");
  HSA_CHECK(scores || total_rows == 0, HSA_ERR_INVALID_ARG, "null scores");
  HSA_CHECK(aligned(offsets, 8) && aligned(scores, 4) && aligned(idx, 4) && aligned(vals, 4),
            HSA_ERR_INVALID_ARG, "misaligned pointer");
  HSA_CHECK(ws && aligned(ws, 256), HSA_ERR_WORKSPACE, "workspace null or not 256-byte aligned");
  HSA_CHECK(ws_bytes >= topk_workspace_bytes(B, total_rows, k), HSA_ERR_WORKSPACE,
            "workspace %zu bytes < %zu needed", ws_bytes, topk_workspace_bytes(B, total_rows, k));
  Spans sp{offsets, nullptr, 0, 1, total_rows};
  return cuda_status(launch_topk(scores, sp, static_cast<int>(B), total_rows, static_cast<int>(k),
                                 idx, vals, ws, static_cast<uint32_t*>(ws),
                                 static_cast<cudaStream_t>(stream)),
                     "topk launch");
}

}  // extern "C"
