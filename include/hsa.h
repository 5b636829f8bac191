/*
 * hsa.h — C ABI of the GB300 (sm_103a) decode-time hybrid sparse-attention library.
 *
 * One decode layer pairs a sliding-window (SWA) KV pool with one compressed
 * pool: C4 (every 4 tokens compressed to one entry, attended through a top-k
 * selection) or C128 (every 128 tokens to one entry, attended densely).
 * Sources, cited by page title and section:
 *   [KD] kerneldigest.dev, "DeepSeek-V4: optimización de inferencia y RL para
 *        modelos con atención híbrida y FP4"
 *   [LH] lehuy.net, "DeepSeek-V4: SGLang và Miles mang đến hỗ trợ Day-0 cho suy
 *        luận nhanh và Học tăng cường"
 *   [WK] AI-KOL wiki, "与 SGLang 团队聊 DeepSeek V4:混合注意力的推理与 RL 训练适配"
 *
 * Conventions shared by every entry point
 *   - Every data pointer is a DEVICE pointer to caller-owned memory on the
 *     current CUDA device; the library allocates nothing.  Scratch memory is a
 *     caller-provided workspace of at least the size returned by the matching
 *     *_workspace_size() function, 256-byte aligned, ZERO-FILLED before its
 *     first use (e.g. cudaMemset); every call leaves it zero-filled again
 *     except for the sticky status word (see hsa_workspace_status).
 *   - bf16 tensors are IEEE bfloat16 (uint16 storage), row-major, contiguous,
 *     16-byte aligned.  fp32 and int tensors are contiguous and naturally
 *     aligned (int64 offsets 8-byte aligned).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Arguments are validated on the host before any launch;
 *     an invalid call returns an error and launches nothing.  No host
 *     synchronisation happens inside a call.
 *   - Ragged sequences: `offsets` is int64 [B+1] (device), sequence b owns rows
 *     [offsets[b], offsets[b+1]), N_b = offsets[b+1] - offsets[b];
 *     `total_rows` (host) must equal offsets[B].  Row indices returned by the
 *     library are row-local (0 .. N_b-1).
 *   - Errors the device can only see at run time (an index out of range, a
 *     capacity overflow, a NaN score, a wait that ran out) do not trap: the
 *     kernel skips the offending access and ORs a bit into the workspace's
 *     sticky status word, read back with hsa_workspace_status().
 */
#ifndef HSA_H_
#define HSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HSA_OK = 0,
  HSA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, k <= 0, ... */
  HSA_ERR_UNSUPPORTED = 2,   /* shape outside the compiled kernels (no fallback) */
  HSA_ERR_CUDA = 3,          /* a CUDA runtime call failed; see hsa_last_error_detail() */
  HSA_ERR_DEVICE_BOUNDS = 4, /* device saw an index / length outside its buffer */
  HSA_ERR_TIMEOUT = 5,       /* a device-side wait gave up after its iteration limit */
  HSA_ERR_WORKSPACE = 6,     /* workspace null, too small or misaligned */
  HSA_ERR_NAN = 7            /* a NaN score reached the top-k (result unspecified) */
} hsa_status_t;

typedef enum { HSA_F32 = 0, HSA_BF16 = 1 } hsa_dtype_t;

/* Kind of compressed pool a layer pairs with its window (= compression ratio). */
typedef enum { HSA_LAYER_C4 = 4, HSA_LAYER_C128 = 128 } hsa_layer_kind_t;

/* Sticky device status bits (OR-ed into the workspace status word). */
#define HSA_DEV_BOUNDS 0x1u
#define HSA_DEV_TIMEOUT 0x2u
#define HSA_DEV_NAN 0x4u

/* Human-readable name of a status code (static string). */
const char* hsa_status_string(hsa_status_t s);

/* Detail of the last failing call on this host thread (static thread-local
 * buffer; empty string if none). */
const char* hsa_last_error_detail(void);

/* Library version as major*10000 + minor*100 + patch. */
int hsa_version(void);

/* Reads and clears the sticky device status word at the head of a workspace.
 * Synchronises `stream`.  Returns HSA_OK if no bit was set, else the status
 * matching the lowest set bit; *bits (may be NULL) receives the raw bits. */
hsa_status_t hsa_workspace_status(void* ws, void* stream, uint32_t* bits);

/* ------------------------------------------------------------------------
 * Flash Compressor — [KD] §Arquitectura del Sistema ("Flash Compressor fuses
 * the 5-stage compression chain into one on-chip pass"); [WK] §推理侧优化,
 * Kernel fusion (read -> add -> softmax -> dot -> write).
 *
 * For every complete block n of r consecutive tokens of sequence s and every
 * channel ch:
 *   out[s, n, ch] = sum_{i<r} softmax_i(z[s, n*r+i, ch] + b[i, ch]) * kv[s, n*r+i, ch]
 * (softmax over the block's r positions, per channel; fp32 arithmetic; the
 * fp32 result is written as fp32 or rounded to nearest-even bf16).  A trailing
 * partial block (T mod r tokens) is not compressed.
 *   kv, z : bf16 [S, T, C]     b : fp32 [r, C]     out : [S, T/r, C] of out_dtype
 * Requirements: S, T >= 0; C a positive multiple of 8; 1 <= r <= 4096; every
 * logit z + b finite (masking by a -inf bias is hsa_compress_overlap's).
 * Reads each input byte once; one kernel launch; no workspace.  Blocks of
 * r <= 16 tokens with C <= 768 pass through a shared-memory ring (bulk
 * copies); its waits are bounded (200 ms, which a working GPU does not reach),
 * and one that runs out ends the kernel with the output incomplete: with no
 * status word, that is not reported.
 * ---------------------------------------------------------------------- */
hsa_status_t hsa_compress(const void* kv, const void* z, const float* b, int64_t S, int64_t T,
                          int64_t C, int64_t r, void* out, int out_dtype, void* stream);

/* ------------------------------------------------------------------------
 * C4 overlap transform — [WK] §RL 训练侧 ① (neighbouring compressed entries
 * share tokens, so a context-parallel split needs its neighbour's tokens).
 * The pages name it without a definition; the library's reading: entry n is
 * the gated average over the 2r-token window of blocks n-1 and n,
 *   out[s, n, ch] = sum_{i in [i0, 2r)} softmax_i(z[s, n*r-r+i, ch] + b[i, ch])
 *                                        * kv[s, n*r-r+i, ch],
 * i0 = r for n = 0 (no block before it), else 0; b has one row per window
 * position.  Arithmetic, output and requirements as hsa_compress, with
 * 1 <= r <= 2048 and b fp32 [2r, C].  A bias of -inf masks its position (the
 * window's other positions must hold a finite logit).
 * ---------------------------------------------------------------------- */
hsa_status_t hsa_compress_overlap(const void* kv, const void* z, const float* b, int64_t S,
                                  int64_t T, int64_t C, int64_t r, void* out, int out_dtype,
                                  void* stream);

/* ------------------------------------------------------------------------
 * Indexer scores — [KD] §Flujo de Inferencia step 6 and §Arquitectura del
 * Sistema (the DSA indexer whose top-k picks the compressed candidates); [WK]
 * §RL 训练侧 (the attention indexer works like an MoE router).
 *
 * For every compressed entry j of sequence b (rows [offsets[b], offsets[b+1])):
 *   scores[j] = sum_{h<Hi} w[b, h] * max(0, sum_{d<Di} iq[b, h, d] * keys[j, d])
 * bf16 products, fp32 accumulation (tcgen05 tensor cores, fp32 TMEM
 * accumulators), fp32 result at the same row position as the key.
 *   iq : bf16 [B, Hi, Di]   w : fp32 [B, Hi]   keys : bf16 [total_rows, Di]
 *   offsets : int64 [B+1]   scores : fp32 [total_rows]
 * Requirements: 1 <= B <= 4096; 1 <= Hi <= 16; Di in {32, 64, 128}; iq and
 * keys 16-byte aligned.  Rows outside every sequence are not written.  One
 * launch (persistent, two CTAs per SM).
 * Workspace: hsa_indexer_scores_workspace_size() bytes (status word only).
 * ---------------------------------------------------------------------- */
size_t hsa_indexer_scores_workspace_size(void);
hsa_status_t hsa_indexer_scores(const void* iq, const float* w, const void* keys,
                                const int64_t* offsets, int64_t B, int64_t Hi, int64_t Di,
                                int64_t total_rows, float* scores, void* ws, size_t ws_bytes,
                                void* stream);

/* ------------------------------------------------------------------------
 * E4M3 storage of the indexer-key pool — the pages speak of FP8 rollout
 * ([LH] §Hỗ trợ Học tăng cường) and of a 1M-token KV cache under 10 GB ([WK]
 * §DeepSeek V4 的新架构) without fixing a format; the library's format is
 * one row of E4M3 codes ("e4m3fn": bias 7, 3 mantissa bits, largest finite
 * 448, no infinities) with one fp32 scale per row, value = scale * code.
 *
 * hsa_quantize_e4m3: per row of x, amax = max |x|, scales[i] = amax / 448 and
 * codes[i, d] = e4m3(x[i, d] * (448 / amax)), rounded to nearest even and
 * saturated at +-448, every step in binary32; a zero row gets scale 0 and
 * zero codes (a NaN entry gives the NaN code; rows are otherwise finite).
 *   x : fp32 [rows, C]   codes : u8 [rows, C]   scales : fp32 [rows]
 * Requirements: rows >= 0; C a positive multiple of 4; x 16-byte aligned,
 * codes 4-byte aligned.  One launch, no workspace.
 *
 * hsa_indexer_scores_e4m3: the indexer scores over an E4M3 key pool, on the
 * dequantized operands: each query row iq[b, h, :] is quantized as above
 * inside the kernel (qhat = sq * code), khat[j] = key_scales[j] * keys[j], and
 *   scores[j] = sum_{h<Hi} w[b, h] * max(0, qhat[b, h, :] . khat[j, :])
 * computed as key_scales[j] * sum_h (w[b, h] sq[b, h]) max(0, codes . codes):
 * E4M3 tensor-core products (tcgen05 kind::f8f6f4), fp32 accumulation.
 *   iq : bf16 [B, Hi, Di]   w : fp32 [B, Hi]   keys : u8 [total_rows, Di]
 *   key_scales : fp32 [total_rows]   offsets : int64 [B+1]   scores : fp32 [total_rows]
 * Requirements as hsa_indexer_scores, with Di = 128; keys 16-byte aligned.
 * Workspace: hsa_indexer_scores_workspace_size() bytes.
 * ---------------------------------------------------------------------- */
hsa_status_t hsa_quantize_e4m3(const float* x, int64_t rows, int64_t C, uint8_t* codes,
                               float* scales, void* stream);

/* ------------------------------------------------------------------------
 * Bounded waits.  Every spin of a kernel on a barrier gives up after a bound
 * (default 2^24 polls or 200 ms), sets HSA_DEV_TIMEOUT in the workspace's
 * status word and stops the kernel: each role leaves its loop, the copies and
 * tensor-core operations already issued are waited for (with the default
 * bound), TMEM is freed and the kernel returns, so the stream and the context
 * stay usable.  hsa_set_wait_limit sets the bound of the indexer kernels'
 * pipeline waits for every later launch in the process (nanos and polls, the
 * first check being a non-blocking test; 0 restores the default of either) so
 * that the abort path can be exercised: with polls = 1 a wait whose phase is
 * not complete at its first check runs out.  Always returns HSA_OK.
 * ---------------------------------------------------------------------- */
hsa_status_t hsa_set_wait_limit(uint64_t nanos, uint32_t polls);
hsa_status_t hsa_indexer_scores_e4m3(const void* iq, const float* w, const uint8_t* keys,
                                     const float* key_scales, const int64_t* offsets, int64_t B,
                                     int64_t Hi, int64_t Di, int64_t total_rows, float* scores,
                                     void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Lightning TopK — [KD] §Arquitectura del Sistema (radix-select reduction in
 * place of a global sort for the indexer's top-k); [WK] §推理侧优化, Lightning
 * topk.
 *
 * Per sequence b, the first min(k, N_b) row-local indices of the scores
 * ordered by value descending, lower index first among equal values (-0.0
 * equals +0.0; +-inf are ordinary values); remaining slots get -1 (idx) and
 * -inf (vals).  Bit-exact: the result depends only on the fp32 scores.
 * A NaN score is a precondition violation: the output is unspecified and the
 * status bit HSA_DEV_NAN is set; nothing faults.
 *   scores : fp32 [total_rows]   offsets : int64 [B+1]
 *   idx : int32 [B, k]   vals : fp32 [B, k] or NULL
 * Requirements: 1 <= k <= 2048; B >= 1.
 * Method: radix select on order-preserving uint32 keys.  When total_rows <=
 * 32768, one launch: a cluster of four CTAs per row holds the row in
 * registers, sums its histogram of the top 11 key bits through distributed
 * shared memory, compacts the keys at or above the threshold bin, and CTA 0
 * settles the boundary and sorts.  Otherwise also one launch, every row cut
 * into chunks handled by separate CTAs: each CTA reads its chunk once and
 * counts (12-bit digits) and keeps only the keys at or above a bar that
 * rises as it reads (the threshold bin of the scores it has seen, which never
 * lies above the row's); the row's last CTA to finish sums the counts, finds
 * the threshold bin, gathers the kept keys, settles the boundary by a radix
 * select over that bin, sorts the k survivors and writes them.
 * ---------------------------------------------------------------------- */
size_t hsa_topk_workspace_size(int64_t B, int64_t total_rows, int64_t k);
hsa_status_t hsa_topk(const float* scores, const int64_t* offsets, int64_t B, int64_t total_rows,
                      int64_t k, int32_t* idx, float* vals, void* ws, size_t ws_bytes,
                      void* stream);

/* ------------------------------------------------------------------------
 * Allocation-free top-k.  The pages have no counterpart to this entry point;
 * it exists for callers that own only their input and output buffers and
 * cannot provide a workspace — code running inside a host framework whose
 * allocator owns all device memory, or a latency-critical path that must not
 * call cudaMalloc (which can synchronise the device).
 *
 * Same arguments, result and requirements as hsa_topk, without the
 * workspace: the scratch lives in a file-scope device array of 16 MiB that
 * every GPU which loads the library holds until the process exits.  A call
 * whose hsa_topk_workspace_size(B, total_rows, k) exceeds 16 MiB is rejected
 * with HSA_ERR_UNSUPPORTED before any launch (e.g. B = 64 rows fit up to
 * about 1.9 million scores in total).  The call allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 * The first call on a device, with that device current, looks up the array's
 * device address (cudaGetSymbolAddress); make that first call before any
 * stream capture.  The address is cached per device with the id of the CUDA
 * context it was taken in, and looked up again (the same way) when that
 * context has changed, e.g. after cudaDeviceReset.  Every call shares the one array and clears the part that
 * must start at zero (a cudaMemsetAsync on `stream`) before its two kernel
 * launches; calls that overlap on the same GPU (e.g. issued on different
 * streams) race on it (each device has its own array).  Device-side status
 * bits (NaN, bad offsets) are not reported by this entry point.
 * ---------------------------------------------------------------------- */
hsa_status_t hsa_topk_noalloc(const float* scores, const int64_t* offsets, int64_t B,
                              int64_t total_rows, int64_t k, int32_t* idx, float* vals,
                              void* stream);

/* ------------------------------------------------------------------------
 * Fused hybrid attention — [KD] §Flujo de Inferencia step 5 and the
 * technology table (FlashMLA: SWA + C4/C128 attention fused in one kernel);
 * [LH] §Tích hợp Kernel (SWA and the extra attention in one kernel call);
 * [WK] §核心观点 (SWA sees the latest tokens, C4 attends its top-k, C128
 * attends everything).
 *
 * For query token b (one per sequence) and head h, the attended slots are
 *   - the window rows of positions p in [max(0, L_b - W), L_b), L_b =
 *     seq_len[b], read from ring slot p mod W of swa[b], and
 *   - sparse (extra_idx != NULL): the compressed rows extra[offsets[b] + j]
 *     for every listed j = extra_idx[b, i], i < k, with j >= 0 (one term per
 *     listed entry; -1 lists nothing; j >= N_b is skipped and sets
 *     HSA_DEV_BOUNDS), or
 *   - dense (extra_idx == NULL): every compressed row of the sequence,
 *     N_b = offsets[b+1] - offsets[b] <= max_extra_rows (excess rows are
 *     skipped and set HSA_DEV_BOUNDS).
 * Keys are the full Dqk-wide rows, values their first Dv channels (one shared
 * latent KV head).  One softmax runs over all slots:
 *   o[b,h,:] = sum_t softmax_t(scale * q[b,h,:] . K_t) * K_t[0:Dv]
 *   lse[b,h] = log sum_t exp(scale * q[b,h,:] . K_t)          (natural log)
 * bf16 MMA inputs (tcgen05), fp32 accumulation and softmax; P is rounded to
 * bf16 for the second product.  A sequence with no slot gives o = 0, lse = -inf.
 *   q : bf16 [B, Hq, Dqk]      swa : bf16 [B, W, Dqk] (may be NULL if W == 0)
 *   seq_len : int32 [B]        extra : bf16 [extra_total_rows, Dqk] or NULL
 *   extra_offsets : int64 [B+1]   extra_idx : int32 [B, k] or NULL
 *   out : [B, Hq, Dv] of out_dtype     lse : fp32 [B, Hq] or NULL
 * Requirements: Hq <= 32 or a multiple of 32; Dqk a multiple of 64 in
 * [128, 576]; Dv a multiple of 128 in [128, Dqk]; q, swa, extra, out
 * 16-byte aligned.  Workspace: hsa_decode_attn_workspace_size(B, Hq, Dqk, Dv,
 * W, extra_slots) with extra_slots = k (sparse) or max_extra_rows (dense);
 * long slot lists are split across S CTAs; with 2 <= S <= 4 the splits of a
 * token form one thread-block cluster and merge in distributed shared memory
 * (the workspace is then the 256-byte header alone), otherwise their fp32
 * partials go through the workspace and a second launch merges them.
 * ---------------------------------------------------------------------- */
size_t hsa_decode_attn_workspace_size(int64_t B, int64_t Hq, int64_t Dqk, int64_t Dv, int64_t W,
                                      int64_t extra_slots);
hsa_status_t hsa_decode_attn(const void* q, const void* swa, const int32_t* seq_len, int64_t W,
                             const void* extra, const int64_t* extra_offsets,
                             int64_t extra_total_rows, const int32_t* extra_idx, int64_t k,
                             int64_t max_extra_rows, int64_t B, int64_t Hq, int64_t Dqk,
                             int64_t Dv, float scale, void* out, int out_dtype, float* lse,
                             void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * One decode step of one hybrid layer — [WK] §核心观点 (each layer keeps the
 * SWA window, its compressed pool and the in-flight block that is compressed
 * once 4 / 128 tokens have accumulated; C4 picks its top-k, C128 attends
 * all); [KD] §Arquitectura del Sistema (compression-state ring buffers) and
 * §Flujo de Inferencia steps 3, 5, 6.
 *
 * With L_b = seq_len_in[b] + 1 (the context after this step's token), in
 * stream order and without host synchronisation:
 *   1. append: kv_new[b] -> swa[b, (L_b-1) mod W]; kv_new, z_new ->
 *      kv_ring / z_ring[b, (L_b-1) mod r]; (C4) ik_new, iz_new -> ik_ring /
 *      iz_ring likewise; seq_len_out[b] = L_b (seq_len_out may alias
 *      seq_len_in: then repeated calls advance the sequence);
 *   2. if L_b mod r == 0: compress the completed ring block (hsa_compress
 *      arithmetic, bf16 result) into kv_pool row pool_offsets[b] + L_b/r - 1
 *      and (C4) the indexer-key ring into key_pool at the same row;
 *   3. (C4) indexer scores over the N_b = L_b/4 live pool rows;
 *   4. (C4) top-k of those scores (topk_idx, row-local, -1 padded);
 *   5. attention over the window and the selected (C4) or all N_b = L_b/128
 *      (C128) pool rows -> out, lse.
 * r = kind.  Pools use a capacity layout: sequence b owns rows
 * [pool_offsets[b], pool_offsets[b+1]) of kv_pool (and key_pool), of which
 * the first L_b / r are live; a step that would write past the capacity sets
 * HSA_DEV_BOUNDS and skips that write.  Rings hold r rows per sequence, in
 * block order.  Kernel launches (hsa_layer_decode_launches gives the count):
 * C4 three (the top-k inside the attention kernel), or four with the top-k
 * on its own (rows above the fused selection's limit); C128 two; one more
 * when the attention's key splits are merged by their own kernel.
 * Consecutive launches overlap under programmatic dependent launch, with the
 * results of the stream order above.
 * Shapes as for the individual stages; C4 needs Hi, Di, k, iq, w, key_pool,
 * the ik / iz rings and b_ik; C128 needs max_pool_rows >= every N_b.
 * ---------------------------------------------------------------------- */
typedef struct hsa_layer_desc {
  int32_t kind;             /* HSA_LAYER_C4 or HSA_LAYER_C128 */
  int32_t B, Hq, Dqk, Dv;   /* sequences, query heads, key / value widths */
  int32_t Hi, Di;           /* indexer heads and width (C4) */
  int32_t W, k;             /* window rows; top-k (C4) */
  float scale;              /* softmax scale */
  int32_t out_dtype;        /* HSA_BF16 or HSA_F32 */
  int64_t pool_total_rows;  /* rows of kv_pool / key_pool */
  int64_t max_pool_rows;    /* bound on live pool rows per sequence: required for C128
                               (dense attention); for C4 an optional hint (0 = unknown)
                               that lets the top-k finish in one clustered launch when
                               <= 32768; a row above the bound is flagged and treated
                               as empty */
  const int32_t* seq_len_in;    /* [B] tokens before this step */
  int32_t* seq_len_out;         /* [B] tokens after this step (may alias) */
  const int64_t* pool_offsets;  /* [B+1] capacity layout of the pools */
  const void* kv_new;       /* bf16 [B, Dqk] new token's latent kv row */
  const void* z_new;        /* bf16 [B, Dqk] its gate logits */
  const float* b_kv;        /* fp32 [r, Dqk] positional gate bias */
  const void* ik_new;       /* bf16 [B, Di] new raw indexer key (C4) */
  const void* iz_new;       /* bf16 [B, Di] its gate logits (C4) */
  const float* b_ik;        /* fp32 [r, Di] (C4) */
  void* swa;                /* bf16 [B, W, Dqk] window ring */
  void* kv_ring;            /* bf16 [B, r, Dqk] in-flight block */
  void* z_ring;             /* bf16 [B, r, Dqk] */
  void* ik_ring;            /* bf16 [B, r, Di] (C4) */
  void* iz_ring;            /* bf16 [B, r, Di] (C4) */
  void* kv_pool;            /* bf16 [pool_total_rows, Dqk] */
  void* key_pool;           /* bf16 [pool_total_rows, Di] (C4) */
  const void* q;            /* bf16 [B, Hq, Dqk] */
  const void* iq;           /* bf16 [B, Hi, Di] (C4) */
  const float* w;           /* fp32 [B, Hi] (C4) */
  void* out;                /* [B, Hq, Dv] of out_dtype */
  float* lse;               /* fp32 [B, Hq] or NULL */
  int32_t* topk_idx;        /* int32 [B, k] or NULL (kept in the workspace) (C4) */
  float* scores;            /* fp32 [pool_total_rows] or NULL (workspace) (C4) */
  void* const* stage_events;  /* NULL, or 5 caller-created cudaEvent_t recorded on `stream`
                                 before the append kernel, after it, after the indexer,
                                 after the top-k and after the attention (C128 records
                                 events 2 and 3 at the same point as event 1).  Kernels
                                 separated by an event do not overlap their launches. */
  void* q_ready_event;      /* NULL, or a caller-created cudaEvent_t that `stream` waits
                               for right before the attention kernel, the only reader of
                               q: q may then still be arriving (e.g. copied from the host
                               on another stream) while the append, indexer and top-k
                               run — [KD] §Arquitectura del Sistema (multi-stream overlap).
                               The attention is then launched without programmatic
                               dependent launch. */
  int32_t key_fp8;          /* (C4) 0: key_pool holds bf16 rows; 1: key_pool holds E4M3
                               codes u8 [pool_total_rows, Di] with key_scale (Di = 128):
                               step 2 quantizes the completed block's fp32 key as
                               hsa_quantize_e4m3 does and step 3 is
                               hsa_indexer_scores_e4m3 */
  float* key_scale;         /* fp32 [pool_total_rows] when key_fp8, else ignored */
  int32_t T;                /* query tokens per sequence in this step (0 or 1: one; at most
                               4; C4: T * Hi <= 16) — speculative decoding with a one-layer
                               multi-token-prediction head verifies the current token and a
                               draft token together ([LH] §Tích hợp Kernel và Giải mã suy
                               đoán), T = 2.  The step appends the T tokens in order
                               (positions L_in .. L_in + T - 1) and token t attends exactly
                               what it would see had the tokens been decoded one per step:
                               the window positions [L_t - W, L_t), L_t = L_in + t + 1, and
                               the L_t / r entries completed up to its position (C4: its own
                               scores and top-k).  With T > 1 the per-token tensors gain a
                               token axis after the batch axis: q [B, T, Hq, Dqk], kv_new /
                               z_new [B, T, Dqk], ik_new / iz_new [B, T, Di], iq
                               [B, T, Hi, Di], w [B, T, Hi], out [B, T, Hq, Dv], lse
                               [B, T, Hq], topk_idx [B, T, k], scores [T, pool_total_rows];
                               the window ring holds W + T - 1 rows per sequence
                               (swa [B, W + T - 1, Dqk], slot = position mod (W + T - 1));
                               seq_len_out = seq_len_in + T */
} hsa_layer_desc;

size_t hsa_layer_decode_workspace_size(const hsa_layer_desc* d);
/* Kernel launches one hsa_layer_decode call with this descriptor makes (0 if
 * the descriptor is invalid). */
int32_t hsa_layer_decode_launches(const hsa_layer_desc* d);
hsa_status_t hsa_layer_decode(const hsa_layer_desc* d, void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* HSA_H_ */
