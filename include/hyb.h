/*
 * hyb.h -- C ABI of libhyb.so: the per-layer attention hot path of hybrid models
 * that interleave Full Attention layers (paged KV cache) with Linear Attention
 * layers (fixed-size recurrent state), on one NVIDIA GB300 (sm_103a).
 *
 * Pages the operations come from:
 *   [KV] "推理框架适配Hybrid Model：KV Cache管理与算子调度实战" (icman.com.cn/news/43047)
 *   [VL] "Hybrid Model推理适配：vLLM与SGLang的工程实践指南"   (gsyq.cn/news/436086)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers are DEVICE pointers unless a comment says "host". The caller
 *   allocates and owns every buffer (inputs, outputs, caches, state pools,
 *   tables, workspace). The library never allocates or frees device memory and
 *   never synchronises the stream; every launch is asynchronous on `stream`
 *   (a cudaStream_t passed as void*; NULL = the legacy default stream).
 * - Host-side argument checks run before any launch; on failure nothing is
 *   launched and HYB_ERR_INVALID_ARG / HYB_ERR_UNSUPPORTED is returned. A failed
 *   launch returns HYB_ERR_CUDA.
 * - Checks that need device data (block ids, slots, state-slot indices read from
 *   device tables) are made by the kernels: an offending access is skipped (never
 *   performed) and a bit is OR-ed into a per-device status word that
 *   hyb_device_status() reads. Kernels never trap, and every device-side wait is
 *   bounded (on expiry the kernel sets HYB_DEVERR_TIMEOUT and returns).
 * - Element types: HYB_BF16 (raw bf16) or HYB_F32. q/k/v/out and the KV caches of
 *   one call share that type. Linear states are always fp32 [KV §2.3].
 * - Data buffers (q, k, v, out, caches, state pools, workspace) must be 16-byte
 *   aligned; index arrays must be aligned to their element size.
 *
 * Layouts
 * -------
 *   packed rows q, k, v, out  [T][H][D], row t = token t (decode: T = B)
 *   paged K cache, V cache    [num_blocks][H][bs][D], bs = block_size: 16 [KV §2.1], 32 [VL],
 *                             or any power of two from 16 to 256
 *                             element (blk, h, s, d) at ((blk*H + h)*bs + s)*D + d
 *   block_tables              int32 [B][max_blocks_per_seq]; logical -> physical block
 *   slot_mapping              int64 [T]; slot = blk*bs + offset; -1 = skip the token
 *   state pool                fp32 [num_slots][H][D][D]; S[i][j], i = key dim, j = value dim
 *   state_slots               int32 [B]; request b uses state pool slot state_slots[b]
 *   cu_q_lens / cu_seqlens    int32 [B+1]; request b owns packed rows [cu[b], cu[b+1])
 *   ctx_lens                  int32 [B]; tokens of request b cached / accumulated before
 *                             this call (its first row sits at absolute position ctx_lens[b])
 */
#ifndef HYB_H_
#define HYB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

typedef enum {
  HYB_OK = 0,
  HYB_ERR_INVALID_ARG = 1,   /* a host-checkable argument is wrong; nothing launched   */
  HYB_ERR_UNSUPPORTED = 2,   /* valid but not built (e.g. a head_dim without a kernel) */
  HYB_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed                   */
  HYB_ERR_DEVICE_CHECK = 4   /* hyb_device_status() found a device-side check set      */
} hyb_status_t;

typedef enum { HYB_F32 = 0, HYB_BF16 = 1, HYB_F16 = 2 } hyb_dtype_t;   /* F16: states only */
typedef enum { HYB_FULL = 0, HYB_LINEAR = 1, HYB_SLIDING = 2 } hyb_layer_type_t;
typedef enum { HYB_MODE_DECODE = 0, HYB_MODE_PREFILL = 1 } hyb_mode_t;

/* bits of the device status word */
#define HYB_DEVERR_BAD_BLOCK     0x1u  /* block id < 0 or >= num_blocks inside a sequence */
#define HYB_DEVERR_BAD_SLOT      0x2u  /* slot >= num_blocks * block_size                 */
#define HYB_DEVERR_BAD_STATE     0x4u  /* state slot < 0 or >= num_state_slots            */
#define HYB_DEVERR_TIMEOUT       0x8u  /* a bounded device-side wait expired              */
#define HYB_DEVERR_MISALIGNED    0x10u /* prefill start not on a chunk boundary           */
#define HYB_DEVERR_BAD_LENGTH    0x20u /* a length exceeds the bound given on the host    */

/* Dimensions of a Full-attention layer and its paged cache. */
typedef struct {
  int32_t num_heads;           /* H (query heads = KV heads; the pages use one H)      */
  int32_t head_dim;            /* D                                                     */
  int32_t block_size;          /* bs: 16 [KV §2.1], 32 [VL]; a power of two, 16..256   */
  int32_t num_blocks;          /* physical blocks in each of the K and V pools          */
  int32_t max_blocks_per_seq;  /* columns of block_tables                               */
  int32_t dtype;               /* hyb_dtype_t of q/k/v/out and of the caches            */
  float scale;                 /* softmax scale (the pages give none; 1/sqrt(D) usual)  */
  int32_t window;              /* 0: every earlier key; W > 0: sliding window, a query  */
                               /* at position i sees keys p with i - W < p <= i         */
} hyb_attn_dims_t;

/* Sliding window [KV §1.3: rewriting the model to sliding-window attention is one of
 * the routes the page lists]. With d->window = W > 0 the decode and prefill calls below
 * attend only to the last W positions up to and including the query's own. Entries of
 * block_tables for blocks that end before the window of a request's earliest query in
 * the call are never read: an allocator may release those blocks and store -1 there. */

/* -------------------------------------------------------------------------
 * A1. Slot mapping [KV §2.1: fixed-size token blocks reached through a page table].
 * For packed row t of request b (cu_q_lens[b] <= t < cu_q_lens[b+1]) at absolute
 * position p = ctx_lens[b] + (t - cu_q_lens[b]):
 *     slot_mapping[t] = block_tables[b][p / bs] * bs + p % bs
 * A negative block id yields slot -1. p / bs >= max_blocks_per_seq or a block id
 * >= num_blocks sets HYB_DEVERR_BAD_BLOCK and yields -1. ctx_lens may be NULL (all 0).
 * Decode is the case cu_q_lens = {0,1,...,B}, ctx_lens = seq_lens - 1.
 * ------------------------------------------------------------------------- */
hyb_status_t hyb_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables,
                              const int32_t* cu_q_lens, const int32_t* ctx_lens, int32_t B,
                              int32_t T, const hyb_attn_dims_t* d, void* stream);

/* -------------------------------------------------------------------------
 * A2. KV append [KV §2.1: every token's key and value vectors are kept].
 * For each t < T with slot s = slot_mapping[t] >= 0 and every head h, copies
 * k[t][h][:] to k_cache[s/bs][h][s%bs][:] and v likewise (bitwise). s >= num_blocks*bs
 * sets HYB_DEVERR_BAD_SLOT and is skipped. T = 0 is a no-op.
 * ------------------------------------------------------------------------- */
hyb_status_t hyb_paged_kv_append(const void* k, const void* v, const int64_t* slot_mapping,
                                 int32_t T, void* k_cache, void* v_cache,
                                 const hyb_attn_dims_t* d, void* stream);

/* -------------------------------------------------------------------------
 * A3. Paged decode attention [KV §2.3: decode uses a PagedAttention-type kernel
 * over Q, K, V and the block table; KV §2.1: cost O(S x D) per step].
 * For each request b and head h, with n = seq_lens[b] (which already counts the
 * token appended this step):
 *     out[b][h][:] = sum_{p<n} softmax_p(scale * q[b][h].K_p) V_p
 * where K_p, V_p are read at block_tables[b][p/bs], offset p%bs. n = 0 gives zeros.
 * d->window = W > 0 restricts p to n - W <= p < n (see "Sliding window" above).
 * max_seq_len (host) must be >= every seq_lens[b]; a longer sequence sets
 * HYB_DEVERR_BAD_LENGTH and is truncated. The kernel splits each sequence into
 * ranges of blocks (split-K) and merges the partial softmax states; `workspace`
 * holds the partials and must have hyb_paged_attn_decode_workspace_size() bytes
 * (0 is allowed when that size is 0). The result does not depend on how other
 * requests in the batch are split. Limits: B <= 65535, num_heads <= 65535 and
 * max_seq_len <= 2^24 (beyond them: HYB_ERR_UNSUPPORTED, nothing launched).
 * ------------------------------------------------------------------------- */
size_t hyb_paged_attn_decode_workspace_size(int32_t B, int32_t max_seq_len,
                                            const hyb_attn_dims_t* d);
hyb_status_t hyb_paged_attn_decode(void* out, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* block_tables,
                                   const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                                   const hyb_attn_dims_t* d, void* workspace, size_t ws_bytes,
                                   void* stream);

/* -------------------------------------------------------------------------
 * Decode step with the KV append fused in: one launch does what hyb_paged_kv_append(k, v,
 * slot_mapping, T = B, ...) followed by hyb_paged_attn_decode(...) do, for a decode batch
 * (one new token per request, row b of k/v/q). The pages pair the two: the new token's K
 * and V are written into the paged cache [KV §2.1] and the decode attends over the cache
 * including them [KV §2.3]; fusing them removes one launch per Full layer and step.
 * - k, v: [B][H][D] this step's rows; slot_mapping: int64 [B], the cache slot of request b's
 *   new row (-1: none), as hyb_slot_mapping gives it for position seq_lens[b] - 1. NULL
 *   means exactly that: each row goes to position seq_lens[b] - 1 through the block table
 *   (nothing when seq_lens[b] = 0 or that block id is invalid), so the step needs no
 *   separate slot-mapping launch.
 * - Caches are written (only at those slots); everything else is as hyb_paged_attn_decode,
 *   with the same workspace. A slot >= num_blocks * block_size sets HYB_DEVERR_BAD_SLOT and
 *   that row is not written.
 * - The result is bit-identical to the two calls when slot_mapping[b] is -1 or the slot of
 *   position seq_lens[b] - 1. Any other slot still receives the row, but the attention of
 *   that step does not see it there.
 * ------------------------------------------------------------------------- */
hyb_status_t hyb_paged_attn_decode_append(void* out, const void* q, const void* k,
                                          const void* v, const int64_t* slot_mapping,
                                          void* k_cache, void* v_cache,
                                          const int32_t* block_tables, const int32_t* seq_lens,
                                          int32_t B, int32_t max_seq_len,
                                          const hyb_attn_dims_t* d, void* workspace,
                                          size_t ws_bytes, void* stream);

/* -------------------------------------------------------------------------
 * Paged decode without a workspace. The pages have no counterpart to this entry point:
 * it exists for callers that cannot allocate device memory -- a runtime whose device
 * memory is all assigned by its own planner and that gives an op only its input and
 * output buffers, or a latency-critical loop that must not call cudaMalloc because it
 * synchronises the device. Same contract and result as hyb_paged_attn_decode, but the
 * split-K partials live in a 16 MiB array of device memory owned by the library (held
 * by every GPU that loads libhyb.so until the process exits); nothing is allocated.
 * - Returns HYB_ERR_UNSUPPORTED, launching nothing, when the partials would need more
 *   than 16 MiB (hyb_paged_attn_decode_workspace_size() > 16 MiB). A batch with more than
 *   one split of 512 keys needs B x H x ceil(max_seq_len / 512) x (4 D + 8) bytes (with a
 *   window, max_seq_len is capped near the window): at H = 32, D = 128 that allows
 *   B x ceil(max_seq_len / 512) <= 1008, e.g. 64 requests up to 7 680 tokens. The
 *   8 x 131 072-token long-context batch needs ~34 MB and is always rejected here.
 * - Argument errors are reported exactly as hyb_paged_attn_decode reports them (same
 *   checks, before any CUDA call); CUDA failures set hyb_last_cuda_error().
 * - The first call on a device looks up the array's device address (with that device
 *   current); make that first call before any stream capture on the device. The address
 *   is cached for the life of the process: after cudaDeviceReset on that device it is
 *   stale and this entry point must not be called again (the device status word that
 *   every entry point uses is cached the same way).
 * - All calls on a device share the array and it keeps the previous call's contents
 *   (nothing in it needs to start at zero). Calls whose kernels overlap on the GPU race
 *   on it: issue them one after another on one stream.
 * ------------------------------------------------------------------------- */
hyb_status_t hyb_paged_attn_decode_noalloc(void* out, const void* q, const void* k_cache,
                                           const void* v_cache, const int32_t* block_tables,
                                           const int32_t* seq_lens, int32_t B,
                                           int32_t max_seq_len, const hyb_attn_dims_t* d,
                                           void* stream);

/* -------------------------------------------------------------------------
 * A4. Causal prefill attention [KV §2.3: prefill uses a FlashAttention-type kernel].
 * Packed row t of request b sits at absolute position i = ctx_lens[b] + (t - cu_q_lens[b])
 * and attends to every cached position p <= i of its request:
 *     out[t][h][:] = sum_{p<=i} softmax_p(scale * q[t][h].K_p) V_p
 * K/V are read from the paged cache, so the call's own rows must be appended first
 * (hyb_paged_kv_append) and a cached prefix (ctx_lens[b] > 0) is attended to as well.
 * d->window = W > 0 restricts p to i - W < p <= i (see "Sliding window" above).
 * ctx_lens may be NULL (all 0). T (host) = cu_q_lens[B], the rows of q and out;
 * max_q_len (host) >= every request's row count.
 * bf16 with D = 128 runs the tensor-core kernel; other supported (dtype, D) pairs run
 * a CUDA-core kernel with the same contract.
 * ------------------------------------------------------------------------- */
hyb_status_t hyb_paged_attn_prefill_causal(void* out, const void* q, const void* k_cache,
                                           const void* v_cache, const int32_t* block_tables,
                                           const int32_t* cu_q_lens, const int32_t* ctx_lens,
                                           int32_t B, int32_t T, int32_t max_q_len,
                                           const hyb_attn_dims_t* d, void* stream);

/* -------------------------------------------------------------------------
 * A5. Linear attention decode step [KV §2.1: S <- S + k (outer) v, output q.S;
 * KV §2.3: inputs Q, K, V and the previous state, outputs the output and the new
 * state; the state is read and updated, never re-zeroed, during decode].
 * For each request b and head h, with S = state_pool[state_slots[b]][h] (fp32, in place):
 *     S[i][j] <- S[i][j] + k[b][h][i] * v[b][h][j]        (one fp32 fma per element)
 *     out[b][h][j] = sum_i q[b][h][i] * S[i][j]           (after the update)
 * A slot outside [0, num_state_slots) sets HYB_DEVERR_BAD_STATE and that request is
 * skipped. Two requests of one call must not share a slot.
 * ------------------------------------------------------------------------- */
hyb_status_t hyb_linear_attn_step(void* out, const void* q, const void* k, const void* v,
                                  float* state_pool, int32_t num_state_slots,
                                  const int32_t* state_slots, int32_t B, int32_t H, int32_t D,
                                  int32_t dtype, void* stream);

/* -------------------------------------------------------------------------
 * Linear decode step with a 16-bit state pool (state-precision study). The pages
 * disagree on the state's precision: [KV §2.3] keeps it in fp32 so that it does not
 * drift over long sequences, while the vLLM/SGLang page stores it in fp16. This entry
 * point exists to measure that trade: same contract as hyb_linear_attn_step, but
 * state_pool holds state_dtype = HYB_BF16 or HYB_F16 elements ([num_slots][H][D][D],
 * 16-bit each, 16-byte aligned), and each element is updated as
 *     S[i][j] <- round16(fmaf(k[i], v[j], float(S[i][j])))      (round to nearest even)
 *     out[j]  = sum_i q[i] * float(S[i][j])                      (after the update)
 * Half the state bytes of the fp32 step, at the cost of rounding every update to 8 (bf16)
 * or 11 (fp16) significant bits. fp32 (hyb_linear_attn_step) is the path the pages
 * prescribe; this one is for comparison.
 * ------------------------------------------------------------------------- */
hyb_status_t hyb_linear_attn_step_lowp(void* out, const void* q, const void* k, const void* v,
                                       void* state_pool, int32_t state_dtype,
                                       int32_t num_state_slots, const int32_t* state_slots,
                                       int32_t B, int32_t H, int32_t D, int32_t dtype,
                                       void* stream);

/* -------------------------------------------------------------------------
 * A6. Linear attention chunked prefill [KV §2.3: state zeroed at request start and
 * accumulated through prefill; KV §2.4: chunks carry the state and chunk boundaries
 * of all layers of a request are aligned].
 * Request b owns rows [cu_seqlens[b], cu_seqlens[b+1]); its starting state is zero
 * when reset[b] != 0 (reset may be NULL: no reset), else state_pool[state_slots[b]].
 * Chunks are the position ranges [c*C, (c+1)*C). Per chunk, with S the state at its
 * start:  O_c = Q_c S + tril(Q_c K_c^T) V_c,   S <- S + K_c^T V_c.
 * This equals hyb_linear_attn_step applied token by token. The final state is written
 * back to the slot. A call must start on a chunk boundary: when ctx_lens is given,
 * ctx_lens[b] % chunk_size != 0 sets HYB_DEVERR_MISALIGNED and request b is skipped.
 * T (host) = cu_seqlens[B], the rows of q/k/v/out; max_len (host) >= every request's
 * row count. chunk_size 64 with D = 128 and bf16
 * runs the tensor-core kernel; other (D, dtype, chunk) combinations run the CUDA-core
 * kernel (same contract).
 * The tensor-core kernel is a cooperative launch of at most one CTA per SM that shares all
 * (request, head) chains' chunks out evenly; a chain cut between two CTAs is handed over
 * through its own state slot, announced by a flag that names the call (a per-call epoch,
 * bumped by a one-thread kernel launched just before, and the launch's grid id). The epoch
 * and the flags live in `workspace` (device memory, 8-byte aligned, at least
 * hyb_linear_attn_chunked_prefill_workspace_size() bytes, owned by the caller; its contents
 * need no initialisation and must be left alone between calls). The library keeps no handoff
 * state of its own: calls with distinct workspaces may run at the same time on any streams.
 * Calls that share one workspace must not overlap on the GPU (calls in order on one stream,
 * eager or captured in graphs, never do); if they do, a waiting CTA gives up after ~2 s and
 * sets HYB_DEVERR_TIMEOUT. A flag is only ever accepted from its own call, so overlap never
 * yields a silently wrong state. The CUDA-core kernel ignores the workspace, but it is
 * checked the same way. A missing, misaligned or short workspace is HYB_ERR_INVALID_ARG
 * (nothing launched) when B > 0.
 * ------------------------------------------------------------------------- */
hyb_status_t hyb_linear_attn_chunked_prefill(void* out, const void* q, const void* k,
                                             const void* v, const int32_t* cu_seqlens,
                                             const int32_t* ctx_lens, float* state_pool,
                                             int32_t num_state_slots,
                                             const int32_t* state_slots, const uint8_t* reset,
                                             int32_t B, int32_t T, int32_t max_len, int32_t H,
                                             int32_t D, int32_t chunk_size, int32_t dtype,
                                             void* workspace, size_t ws_bytes, void* stream);

/* Bytes of device workspace hyb_linear_attn_chunked_prefill needs (a fixed 2 056: one
 * 64-bit epoch and one 64-bit flag per CTA, at most 256 CTAs). */
size_t hyb_linear_attn_chunked_prefill_workspace_size(void);

/* -------------------------------------------------------------------------
 * A7. Layer dispatch [KV §2.2: layer types registered from the model config,
 * split memory pools, per-forward metadata of seq lens, block tables and state
 * buffers handed to each op together with the layer type; VL §3.2: an execution
 * plan built per layer type; VL §5.2: each layer has its own cache].
 * layer_types (host, [L]) holds HYB_FULL / HYB_LINEAR / HYB_SLIDING. layers (host, [L]) gives
 * each layer's own buffers; meta (host struct of device pointers) is shared by all
 * layers of the batch. Layers run in order on `stream`:
 *   decode  (mode 0): FULL   -> hyb_paged_attn_decode_append(k, v @ slot_mapping,
 *                               seq_lens): the append and the decode in one launch;
 *                               meta->slot_mapping may be NULL (position seq_lens[b] - 1)
 *                     LINEAR -> hyb_linear_attn_step(state_slots)
 *   prefill (mode 1): FULL   -> hyb_paged_kv_append + hyb_paged_attn_prefill_causal
 *                     LINEAR -> hyb_linear_attn_chunked_prefill(reset, chunk_size)
 * A SLIDING layer runs as a FULL layer with window = layers[l].window (> 0); FULL
 * layers attend to every earlier key, and d->window must be 0.
 * Every layer's arguments are checked before the first launch. Results equal the
 * per-op calls bit for bit. In decode mode the layers overlap at their boundaries: a layer
 * after the first reads its inputs (q/k/v, cache or state pool, the block table, seq_lens
 * and the slot mapping) and does its main work before the previous layer's kernels have
 * finished, and writes the shared workspace only after. No kernel of the dispatch writes
 * those inputs, so this is exact as long as no layer's out aliases another layer's q/k/v,
 * cache, state pool or the batch metadata (which the caller must not do anyway). workspace serves the decode calls (see A3) and must hold
 * hyb_paged_attn_decode_workspace_size() bytes for the largest window among the layers
 * (window 0 when any FULL layer is present). In prefill mode it serves the LINEAR layers'
 * chunked prefill instead (one after another in stream order, sharing it) and must hold
 * hyb_linear_attn_chunked_prefill_workspace_size() bytes when a LINEAR layer is present.
 * ------------------------------------------------------------------------- */
typedef struct {
  void* out;                 /* [T][H][D]                                   */
  const void* q;             /* [T][H][D]                                   */
  const void* k;             /* [T][H][D]                                   */
  const void* v;             /* [T][H][D]                                   */
  void* k_cache;             /* FULL: this layer's own K pool, else NULL    */
  void* v_cache;             /* FULL: this layer's own V pool, else NULL    */
  float* state_pool;         /* LINEAR: this layer's own state pool         */
  int32_t num_state_slots;   /* LINEAR: slots in state_pool                 */
  int32_t window;            /* SLIDING: its window W > 0; otherwise 0      */
} hyb_layer_io_t;

typedef struct {
  const int32_t* seq_lens;      /* [B] decode: cached length incl. the new token     */
  const int32_t* block_tables;  /* [B][max_blocks_per_seq]                           */
  const int64_t* slot_mapping;  /* [T]                                               */
  const int32_t* cu_q_lens;     /* [B+1] prefill rows per request                    */
  const int32_t* ctx_lens;      /* [B] prefill: tokens before this call (may be NULL) */
  const int32_t* state_slots;   /* [B]                                               */
  const uint8_t* reset;         /* [B] prefill: zero the linear state first (NULL ok) */
  int32_t B;
  int32_t T;                    /* rows per layer (decode: B)                        */
  int32_t max_seq_len;          /* decode bound on seq_lens                          */
  int32_t max_q_len;            /* prefill bound on rows per request                 */
} hyb_batch_meta_t;

hyb_status_t hyb_layer_dispatch(const int32_t* layer_types, int32_t L, int32_t mode,
                                const hyb_layer_io_t* layers, const hyb_batch_meta_t* meta,
                                const hyb_attn_dims_t* d, int32_t chunk_size, void* workspace,
                                size_t ws_bytes, void* stream);

/* -------------------------------------------------------------------------
 * Memory accounting [KV §2.1, §3.3]. All arguments are host values.
 *   full   = 2 * L_full * H * D * tokens * batch * kv_elem_bytes
 *   linear = L_linear * H * D * D * batch * state_elem_bytes
 * Returns full + linear and stores the parts when the pointers (host) are non-NULL.
 * ------------------------------------------------------------------------- */
uint64_t hyb_cache_bytes(int32_t L_full, int32_t L_linear, int32_t H, int32_t D, int64_t tokens,
                         int32_t batch, int32_t kv_elem_bytes, int32_t state_elem_bytes,
                         uint64_t* full_out, uint64_t* linear_out);

/* Bounded-wait self-test (failure detection without a fault). Launches one small kernel
 * on `stream` (NULL: the default stream) whose two device-side waits can never be met: an
 * mbarrier phase that nothing completes (the helper behind every TMA and tensor-core wait
 * in the library) and a global flag that nothing sets (the acquire-load wait of the
 * chunked linear prefill's state handoff). Each gives up after limit_us microseconds and
 * sets HYB_DEVERR_TIMEOUT in the device status word, which hyb_device_status() then
 * reports; the kernel returns normally and the context stays usable.
 * limit_us outside [1, 1000000] returns HYB_ERR_INVALID_ARG before any launch. */
hyb_status_t hyb_selftest_bounded_waits(uint32_t limit_us, void* stream);

/* Reads (and, if clear != 0, zeroes) the device status word of the current device
 * into *flags (host). Synchronises the device. Returns HYB_ERR_DEVICE_CHECK when any
 * bit was set, HYB_OK otherwise. */
hyb_status_t hyb_device_status(uint32_t* flags, int32_t clear);

/* Static description of a status code (never NULL). */
const char* hyb_status_string(hyb_status_t s);

/* Text of the CUDA runtime error behind the last HYB_ERR_CUDA that an entry point returned
 * on this thread ("no error" if none). Never NULL. */
const char* hyb_last_cuda_error(void);

/* Number of kernel launches this library has issued on this thread since the last
 * call with reset != 0 (host-side counter; benchmarks report it). */
uint64_t hyb_launch_count(int32_t reset);

/* Dispatch trace. With HYB_TRACE set in the environment (to anything but "" or "0"),
 * hyb_layer_dispatch writes one line per layer to stderr naming the kernels it launches
 * for that layer, and records a CUDA event before the first layer and after each layer on
 * the dispatch's stream (not while the stream is being captured into a graph). Events are
 * created once per host thread and device and reused; no device memory is allocated.
 * hyb_trace_layer_ms fills ms[0..L0) with each layer's device time in milliseconds for the
 * last traced dispatch of this thread (L0 layers), waiting for its last event; it returns
 * HYB_ERR_INVALID_ARG when there is none, when L < L0, or when the current device differs. */
hyb_status_t hyb_trace_layer_ms(float* ms, int32_t L);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif
#ifdef __cplusplus
}
#endif
#endif /* HYB_H_ */
