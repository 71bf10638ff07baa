// C ABI of libhyb.so: host-side argument checks, launch sequencing and the per-device
// status word. Every operation is defined in include/hyb.h with its page citation.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <set>
#include <utility>
#include <vector>

#include "hyb_internal.cuh"

// Device-side check word (one per device that loads the library); kernels OR bits in.
static __device__ unsigned g_hyb_status;
// A flag that nothing ever sets: the bounded-wait self-test waits on it.
static __device__ unsigned long long g_hyb_never_set;

namespace hyb {
namespace {
// Two device-side waits that nothing satisfies, each with the library's bounded-wait
// mechanism: warp 0 on an mbarrier phase that no thread or copy completes (the helper every
// TMA and tensor-core wait uses), warp 1 on a global flag that no thread sets (an acquire
// load, %globaltimer and a back-off, as in the chunked linear prefill's state handoff). Each
// gives up after limit_ns, reports HYB_DEVERR_TIMEOUT and returns.
__global__ void selftest_bounded_waits_kernel(uint64_t limit_ns, unsigned* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait(&bar, 0, limit_ns)) flag(status, HYB_DEVERR_TIMEOUT);
  } else if (threadIdx.x == 32) {
    const uint64_t t0 = global_ns();
    while (true) {
      unsigned long long v;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(&g_hyb_never_set) : "memory");
      if (v == ~0ull) break;                   // never true: nothing writes the flag
      if (global_ns() - t0 > limit_ns) {
        flag(status, HYB_DEVERR_TIMEOUT);
        break;
      }
      __nanosleep(1000);
    }
  }
}
}  // namespace
}  // namespace hyb

namespace hyb {
namespace {
std::mutex g_mu;
constexpr int kMaxDev = 64;
unsigned* g_status_addr[kMaxDev] = {};
int g_sms[kMaxDev] = {};
std::set<std::pair<const void*, int>> g_smem_done;
thread_local uint64_t g_launches = 0;

int cur_dev() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDev) return -1;
  return d;
}
}  // namespace

void count_launch() { ++g_launches; }

int num_sms() {
  const int d = cur_dev();
  if (d < 0) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[d]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = n > 0 ? n : 1;
  }
  return g_sms[d];
}

cudaError_t set_smem(const void* fn, int bytes) {
  const int d = cur_dev();
  if (d < 0) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_smem_done.count({fn, d})) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) g_smem_done.insert({fn, d});
  return e;
}

// Address of this device's status word (looked up once per device, with it current).
unsigned* status_word() {
  const int d = cur_dev();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_addr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_hyb_status) != cudaSuccess) return nullptr;
    g_status_addr[d] = static_cast<unsigned*>(p);
  }
  return g_status_addr[d];
}

}  // namespace hyb

using namespace hyb;

namespace {

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool al(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline int esize_of(int dtype) { return dtype == HYB_BF16 ? 2 : 4; }

thread_local cudaError_t g_last_cuda = cudaSuccess;

}  // namespace

namespace hyb {

hyb_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return HYB_OK;
  g_last_cuda = e;
  return HYB_ERR_CUDA;
}

hyb_status_t check_dims(const hyb_attn_dims_t* d) {
  if (!d) return HYB_ERR_INVALID_ARG;
  if (d->num_heads <= 0 || d->head_dim <= 0 || d->num_blocks <= 0 || d->max_blocks_per_seq <= 0)
    return HYB_ERR_INVALID_ARG;
  if (!block_size_ok(d->block_size)) return HYB_ERR_UNSUPPORTED;
  if (d->dtype != HYB_BF16 && d->dtype != HYB_F32) return HYB_ERR_INVALID_ARG;
  if ((d->head_dim * esize_of(d->dtype)) % 16 != 0) return HYB_ERR_UNSUPPORTED;
  if (!std::isfinite(d->scale) || d->window < 0) return HYB_ERR_INVALID_ARG;
  // slots and the pool rows the tensor maps address (blocks x heads x tokens) are int32
  if ((int64_t)d->num_blocks * d->num_heads * d->block_size > INT32_MAX) return HYB_ERR_UNSUPPORTED;
  return HYB_OK;
}

hyb_status_t check_decode_args(const void* out, const void* q, const void* kc, const void* vc,
                               const int32_t* bt, const int32_t* seq_lens, int B, int max_seq_len,
                               const hyb_attn_dims_t* d) {
  hyb_status_t st = check_dims(d);
  if (st != HYB_OK) return st;
  if (B < 0 || max_seq_len < 0) return HYB_ERR_INVALID_ARG;
  if (d->num_heads > 65535 || B > 65535) return HYB_ERR_UNSUPPORTED;   // grid.z = heads, grid.y = rows
  if ((int64_t)max_seq_len > (int64_t)d->max_blocks_per_seq * d->block_size) return HYB_ERR_INVALID_ARG;
  if (max_seq_len > (1 << 24)) return HYB_ERR_UNSUPPORTED;   // bounds the split-K workspace
  if (!decode_supported(d->dtype, d->head_dim)) return HYB_ERR_UNSUPPORTED;
  if (B == 0) return HYB_OK;
  if (!out || !q || !kc || !vc || !bt || !seq_lens) return HYB_ERR_INVALID_ARG;
  if (!al16(out) || !al16(q) || !al16(kc) || !al16(vc) || !al(bt, 4) || !al(seq_lens, 4))
    return HYB_ERR_INVALID_ARG;
  return HYB_OK;
}

}  // namespace hyb

namespace {

// ---- per-op checks (no launch) -----------------------------------------------------
hyb_status_t check_append(const void* k, const void* v, const int64_t* slot, int T,
                          const void* kc, const void* vc, const hyb_attn_dims_t* d) {
  hyb_status_t st = check_dims(d);
  if (st != HYB_OK) return st;
  if (T < 0) return HYB_ERR_INVALID_ARG;
  if (T == 0) return HYB_OK;
  if (!k || !v || !slot || !kc || !vc) return HYB_ERR_INVALID_ARG;
  if (!al16(k) || !al16(v) || !al16(kc) || !al16(vc) || !al(slot, 8)) return HYB_ERR_INVALID_ARG;
  if (kc == vc) return HYB_ERR_INVALID_ARG;
  return HYB_OK;
}

hyb_status_t check_decode(const void* out, const void* q, const void* kc, const void* vc,
                          const int32_t* bt, const int32_t* seq_lens, int B, int max_seq_len,
                          const hyb_attn_dims_t* d, const void* ws, size_t ws_bytes) {
  hyb_status_t st = check_decode_args(out, q, kc, vc, bt, seq_lens, B, max_seq_len, d);
  if (st != HYB_OK || B == 0) return st;
  const DecodePlan p = plan_decode(B, d->num_heads, d->head_dim, max_seq_len, d->window);
  if (p.ws_bytes > 0 && (!ws || ws_bytes < p.ws_bytes || !al16(ws))) return HYB_ERR_INVALID_ARG;
  return HYB_OK;
}

hyb_status_t check_prefill(const void* out, const void* q, const void* kc, const void* vc,
                           const int32_t* bt, const int32_t* cu, const int32_t* ctx, int B, int T,
                           int max_q_len, const hyb_attn_dims_t* d) {
  hyb_status_t st = check_dims(d);
  if (st != HYB_OK) return st;
  if (B < 0 || T < 0 || max_q_len < 0 || max_q_len > T) return HYB_ERR_INVALID_ARG;
  if (d->num_heads > 65535 || B > 65535) return HYB_ERR_UNSUPPORTED;
  if ((int64_t)max_q_len > (int64_t)d->max_blocks_per_seq * d->block_size) return HYB_ERR_INVALID_ARG;
  if (!prefill_tc_supported(d->dtype, d->head_dim) && !decode_supported(d->dtype, d->head_dim))
    return HYB_ERR_UNSUPPORTED;
  if (B == 0 || max_q_len == 0) return HYB_OK;
  if (!out || !q || !kc || !vc || !bt || !cu) return HYB_ERR_INVALID_ARG;
  if (!al16(out) || !al16(q) || !al16(kc) || !al16(vc) || !al(bt, 4) || !al(cu, 4) ||
      (ctx && !al(ctx, 4)))
    return HYB_ERR_INVALID_ARG;
  if ((int64_t)B * max_q_len > INT32_MAX) return HYB_ERR_UNSUPPORTED;
  return HYB_OK;
}

// pool_align: 16 for the fp32 pool (float4 rows), 8 for a 16-bit pool (4-element rows)
hyb_status_t check_linear_common(const void* out, const void* q, const void* k, const void* v,
                                 const void* pool, int NS, const int32_t* slots, int B, int H,
                                 int D, int dtype, unsigned pool_align = 16) {
  if (B < 0 || H <= 0 || D <= 0 || NS <= 0) return HYB_ERR_INVALID_ARG;
  if (dtype != HYB_BF16 && dtype != HYB_F32) return HYB_ERR_INVALID_ARG;
  if (B > 65535 || H > 65535) return HYB_ERR_UNSUPPORTED;   // grid.z / grid.y limits
  if (!linear_supported(dtype, D)) return HYB_ERR_UNSUPPORTED;
  if (B == 0) return HYB_OK;
  if (!out || !q || !k || !v || !pool || !slots) return HYB_ERR_INVALID_ARG;
  if (!al16(out) || !al16(q) || !al16(k) || !al16(v) || !al(pool, pool_align) || !al(slots, 4))
    return HYB_ERR_INVALID_ARG;
  if ((int64_t)NS * H * D * D > ((int64_t)1 << 40)) return HYB_ERR_UNSUPPORTED;
  return HYB_OK;
}

hyb_status_t check_linear_prefill(const void* out, const void* q, const void* k, const void* v,
                                  const int32_t* cu, const int32_t* ctx, const float* pool,
                                  int NS, const int32_t* slots, const uint8_t* reset, int B, int T,
                                  int max_len, int H, int D, int C, int dtype, const void* ws,
                                  size_t ws_bytes) {
  hyb_status_t st = check_linear_common(out, q, k, v, pool, NS, slots, B, H, D, dtype);
  if (st != HYB_OK) return st;
  if (C <= 0 || T < 0 || max_len < 0 || max_len > T) return HYB_ERR_INVALID_ARG;
  if (!linear_prefill_tc_supported(dtype, D, C) && D > 128) return HYB_ERR_UNSUPPORTED;
  if (B == 0) return HYB_OK;
  if (!cu || !al(cu, 4) || (ctx && !al(ctx, 4))) return HYB_ERR_INVALID_ARG;
  if (!ws || !al(ws, 8) || ws_bytes < kLinPrefillWsBytes) return HYB_ERR_INVALID_ARG;
  (void)reset;
  return HYB_OK;
}

// ---- launches (arguments already checked) -----------------------------------------
hyb_status_t run_decode(void* out, const void* q, const void* kc, const void* vc,
                        const int32_t* bt, const int32_t* seq_lens, int B, int max_seq_len,
                        const hyb_attn_dims_t* d, void* ws, unsigned* status, cudaStream_t s,
                        const DecodeAppend* app = nullptr, bool early = false) {
  if (B == 0) return HYB_OK;
  const DecodePlan p = plan_decode(B, d->num_heads, d->head_dim, max_seq_len, d->window);
  return cuda_status(launch_paged_decode(out, q, kc, vc, bt, seq_lens, nullptr, nullptr, B, 0,
                                         d->num_heads, d->head_dim, d->dtype, d->num_blocks,
                                         d->max_blocks_per_seq, d->block_size, max_seq_len,
                                         d->scale, d->window, p, ws, status, s, app, early));
}

hyb_status_t run_prefill(void* out, const void* q, const void* kc, const void* vc,
                         const int32_t* bt, const int32_t* cu, const int32_t* ctx, int B, int T,
                         int max_q_len, const hyb_attn_dims_t* d, unsigned* status,
                         cudaStream_t s) {
  if (B == 0 || max_q_len == 0) return HYB_OK;
  if (prefill_tc_supported(d->dtype, d->head_dim))
    return cuda_status(launch_prefill_tc(out, q, kc, vc, bt, cu, ctx, B, T, max_q_len,
                                         d->num_heads, d->num_blocks, d->max_blocks_per_seq,
                                         d->block_size, d->scale, d->window, status, s));
  const DecodePlan none{1 << 30, 1, 0};
  return cuda_status(launch_paged_decode(out, q, kc, vc, bt, nullptr, cu, ctx, B, max_q_len,
                                         d->num_heads, d->head_dim, d->dtype, d->num_blocks,
                                         d->max_blocks_per_seq, d->block_size,
                                         d->max_blocks_per_seq * d->block_size, d->scale,
                                         d->window, none, nullptr, status, s));
}

hyb_status_t run_linear_prefill(void* out, const void* q, const void* k, const void* v,
                                const int32_t* cu, const int32_t* ctx, float* pool, int NS,
                                const int32_t* slots, const uint8_t* reset, int B, int T,
                                int max_len, int H, int D, int C, int dtype, void* ws,
                                unsigned* status, cudaStream_t s) {
  if (B == 0) return HYB_OK;
  if (linear_prefill_tc_supported(dtype, D, C))
    return cuda_status(launch_linear_prefill_tc(out, q, k, v, cu, ctx, pool, NS, slots, reset,
                                                B, T, max_len, H, C, ws, status, s));
  return cuda_status(launch_linear_prefill_simt(out, q, k, v, cu, ctx, pool, NS, slots, reset,
                                                B, H, D, C, dtype, status, s));
}

}  // namespace

extern "C" {

hyb_status_t hyb_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables,
                              const int32_t* cu_q_lens, const int32_t* ctx_lens, int32_t B,
                              int32_t T, const hyb_attn_dims_t* d, void* stream) {
  hyb_status_t st = check_dims(d);
  if (st != HYB_OK) return st;
  if (B < 0 || T < 0) return HYB_ERR_INVALID_ARG;
  if (B == 0 || T == 0) return HYB_OK;
  if (!slot_mapping || !block_tables || !cu_q_lens) return HYB_ERR_INVALID_ARG;
  if (!al(slot_mapping, 8) || !al(block_tables, 4) || !al(cu_q_lens, 4) ||
      (ctx_lens && !al(ctx_lens, 4)))
    return HYB_ERR_INVALID_ARG;
  unsigned* sw = status_word();
  if (!sw) return HYB_ERR_CUDA;
  return cuda_status(launch_slot_mapping(slot_mapping, block_tables, cu_q_lens, ctx_lens, B, T,
                                         d->max_blocks_per_seq, d->num_blocks, d->block_size, sw,
                                         (cudaStream_t)stream));
}

hyb_status_t hyb_paged_kv_append(const void* k, const void* v, const int64_t* slot_mapping,
                                 int32_t T, void* k_cache, void* v_cache,
                                 const hyb_attn_dims_t* d, void* stream) {
  hyb_status_t st = check_append(k, v, slot_mapping, T, k_cache, v_cache, d);
  if (st != HYB_OK || T == 0) return st;
  unsigned* sw = status_word();
  if (!sw) return HYB_ERR_CUDA;
  return cuda_status(launch_kv_append(k, v, slot_mapping, T, d->num_heads, d->head_dim,
                                      esize_of(d->dtype), d->num_blocks, d->block_size, k_cache,
                                      v_cache, sw, (cudaStream_t)stream));
}

size_t hyb_paged_attn_decode_workspace_size(int32_t B, int32_t max_seq_len,
                                            const hyb_attn_dims_t* d) {
  if (!d || B <= 0 || max_seq_len <= 0 || d->num_heads <= 0 || d->head_dim <= 0) return 0;
  if (d->window < 0) return 0;
  return plan_decode(B, d->num_heads, d->head_dim, max_seq_len, d->window).ws_bytes;
}

hyb_status_t hyb_paged_attn_decode(void* out, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* block_tables,
                                   const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                                   const hyb_attn_dims_t* d, void* workspace, size_t ws_bytes,
                                   void* stream) {
  hyb_status_t st = check_decode(out, q, k_cache, v_cache, block_tables, seq_lens, B,
                                 max_seq_len, d, workspace, ws_bytes);
  if (st != HYB_OK || B == 0) return st;
  unsigned* sw = status_word();
  if (!sw) return HYB_ERR_CUDA;
  return run_decode(out, q, k_cache, v_cache, block_tables, seq_lens, B, max_seq_len, d,
                    workspace, sw, (cudaStream_t)stream);
}

hyb_status_t hyb_paged_attn_decode_append(void* out, const void* q, const void* k,
                                          const void* v, const int64_t* slot_mapping,
                                          void* k_cache, void* v_cache,
                                          const int32_t* block_tables, const int32_t* seq_lens,
                                          int32_t B, int32_t max_seq_len,
                                          const hyb_attn_dims_t* d, void* workspace,
                                          size_t ws_bytes, void* stream) {
  // a null slot_mapping means: position seq_lens[b] - 1 through the block table
  static const int64_t dummy_slot = 0;
  hyb_status_t st = check_append(k, v, slot_mapping ? slot_mapping : &dummy_slot, B, k_cache,
                                 v_cache, d);
  if (st != HYB_OK) return st;
  st = check_decode(out, q, k_cache, v_cache, block_tables, seq_lens, B, max_seq_len, d,
                    workspace, ws_bytes);
  if (st != HYB_OK || B == 0) return st;
  unsigned* sw = status_word();
  if (!sw) return HYB_ERR_CUDA;
  const DecodeAppend app{k, v, slot_mapping};
  return run_decode(out, q, k_cache, v_cache, block_tables, seq_lens, B, max_seq_len, d,
                    workspace, sw, (cudaStream_t)stream, &app);
}

hyb_status_t hyb_paged_attn_prefill_causal(void* out, const void* q, const void* k_cache,
                                           const void* v_cache, const int32_t* block_tables,
                                           const int32_t* cu_q_lens, const int32_t* ctx_lens,
                                           int32_t B, int32_t T, int32_t max_q_len,
                                           const hyb_attn_dims_t* d, void* stream) {
  hyb_status_t st = check_prefill(out, q, k_cache, v_cache, block_tables, cu_q_lens, ctx_lens, B,
                                  T, max_q_len, d);
  if (st != HYB_OK || B == 0 || max_q_len == 0) return st;
  unsigned* sw = status_word();
  if (!sw) return HYB_ERR_CUDA;
  return run_prefill(out, q, k_cache, v_cache, block_tables, cu_q_lens, ctx_lens, B, T,
                     max_q_len, d, sw, (cudaStream_t)stream);
}

hyb_status_t hyb_linear_attn_step(void* out, const void* q, const void* k, const void* v,
                                  float* state_pool, int32_t num_state_slots,
                                  const int32_t* state_slots, int32_t B, int32_t H, int32_t D,
                                  int32_t dtype, void* stream) {
  hyb_status_t st = check_linear_common(out, q, k, v, state_pool, num_state_slots, state_slots,
                                        B, H, D, dtype);
  if (st != HYB_OK || B == 0) return st;
  unsigned* sw = status_word();
  if (!sw) return HYB_ERR_CUDA;
  return cuda_status(launch_linear_step(out, q, k, v, state_pool, num_state_slots, state_slots,
                                        B, H, D, dtype, sw, (cudaStream_t)stream));
}

hyb_status_t hyb_linear_attn_step_lowp(void* out, const void* q, const void* k, const void* v,
                                       void* state_pool, int32_t state_dtype,
                                       int32_t num_state_slots, const int32_t* state_slots,
                                       int32_t B, int32_t H, int32_t D, int32_t dtype,
                                       void* stream) {
  if (state_dtype != HYB_BF16 && state_dtype != HYB_F16) return HYB_ERR_INVALID_ARG;
  hyb_status_t st = check_linear_common(out, q, k, v, state_pool, num_state_slots, state_slots,
                                        B, H, D, dtype);   // 16-byte aligned pool
  if (st != HYB_OK || B == 0) return st;
  unsigned* sw = status_word();
  if (!sw) return HYB_ERR_CUDA;
  return cuda_status(launch_linear_step_lowp(out, q, k, v, state_pool, state_dtype,
                                             num_state_slots, state_slots, B, H, D, dtype, sw,
                                             (cudaStream_t)stream));
}

hyb_status_t hyb_linear_attn_chunked_prefill(void* out, const void* q, const void* k,
                                             const void* v, const int32_t* cu_seqlens,
                                             const int32_t* ctx_lens, float* state_pool,
                                             int32_t num_state_slots,
                                             const int32_t* state_slots, const uint8_t* reset,
                                             int32_t B, int32_t T, int32_t max_len, int32_t H,
                                             int32_t D, int32_t chunk_size, int32_t dtype,
                                             void* workspace, size_t ws_bytes, void* stream) {
  hyb_status_t st = check_linear_prefill(out, q, k, v, cu_seqlens, ctx_lens, state_pool,
                                         num_state_slots, state_slots, reset, B, T, max_len, H, D,
                                         chunk_size, dtype, workspace, ws_bytes);
  if (st != HYB_OK || B == 0) return st;
  unsigned* sw = status_word();
  if (!sw) return HYB_ERR_CUDA;
  return run_linear_prefill(out, q, k, v, cu_seqlens, ctx_lens, state_pool, num_state_slots,
                            state_slots, reset, B, T, max_len, H, D, chunk_size, dtype,
                            workspace, sw, (cudaStream_t)stream);
}

size_t hyb_linear_attn_chunked_prefill_workspace_size(void) { return kLinPrefillWsBytes; }

// ---- dispatch trace (HYB_TRACE set in the environment): a line per layer on stderr naming
// its kernels, and a CUDA event before the first layer and after each layer, kept per host
// thread so hyb_trace_layer_ms can report the last traced dispatch.
namespace {
struct Trace {
  std::vector<cudaEvent_t> ev;
  int layers = 0;                          // layers of the last traced dispatch (0: none)
  int dev = -1;
};
thread_local Trace g_trace;

bool trace_on(cudaStream_t s) {
  const char* e = std::getenv("HYB_TRACE");
  if (!e || !*e || (e[0] == '0' && !e[1])) return false;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return false;                          // not inside a graph capture
  return true;
}

// Event i of the current trace (created on first use, on the current device).
cudaEvent_t trace_event(int i) {
  const int d = cur_dev();
  if (d != g_trace.dev) {                  // events belong to a device: start over
    for (cudaEvent_t e : g_trace.ev) cudaEventDestroy(e);
    g_trace.ev.clear();
    g_trace.dev = d;
  }
  while ((int)g_trace.ev.size() <= i) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_trace.ev.push_back(e);
  }
  return g_trace.ev[i];
}

const char* layer_kernels(int lt, int mode, const hyb_attn_dims_t* d, int chunk) {
  if (lt == HYB_LINEAR)
    return mode == HYB_MODE_DECODE ? "linear_step_kernel"
           : linear_prefill_tc_supported(d->dtype, d->head_dim, chunk)
               ? "linear_handoff_epoch_kernel + linear_prefill_tc_kernel"
               : "linear_prefill_simt_kernel";
  if (mode == HYB_MODE_DECODE) return "paged_decode_kernel (KV append fused) [+ decode_combine_kernel]";
  return prefill_tc_supported(d->dtype, d->head_dim) ? "kv_append_kernel + prefill_tc_kernel"
                                                     : "kv_append_kernel + paged_decode_kernel<prefill>";
}
}  // namespace

hyb_status_t hyb_trace_layer_ms(float* ms, int32_t L) {
  if (!ms || g_trace.layers == 0 || L < g_trace.layers) return HYB_ERR_INVALID_ARG;
  if (cur_dev() != g_trace.dev) return HYB_ERR_INVALID_ARG;
  cudaError_t e = cudaEventSynchronize(g_trace.ev[g_trace.layers]);
  for (int l = 0; e == cudaSuccess && l < g_trace.layers; ++l)
    e = cudaEventElapsedTime(&ms[l], g_trace.ev[l], g_trace.ev[l + 1]);
  return cuda_status(e);
}

hyb_status_t hyb_layer_dispatch(const int32_t* layer_types, int32_t L, int32_t mode,
                                const hyb_layer_io_t* layers, const hyb_batch_meta_t* meta,
                                const hyb_attn_dims_t* d, int32_t chunk_size, void* workspace,
                                size_t ws_bytes, void* stream) {
  if (L < 0 || (L > 0 && (!layer_types || !layers)) || !meta || !d) return HYB_ERR_INVALID_ARG;
  if (mode != HYB_MODE_DECODE && mode != HYB_MODE_PREFILL) return HYB_ERR_INVALID_ARG;
  hyb_status_t st = check_dims(d);
  if (st != HYB_OK) return st;
  if (d->window != 0) return HYB_ERR_INVALID_ARG;     // windows come from the layer types
  const int B = meta->B, T = meta->T, H = d->num_heads, D = d->head_dim, dt = d->dtype;
  if (B < 0 || T < 0) return HYB_ERR_INVALID_ARG;
  if (mode == HYB_MODE_DECODE && T != B) return HYB_ERR_INVALID_ARG;
  // 1) check every layer before launching anything
  std::set<const void*> seen;   // each layer owns its caches / state pool [VL §5.2]
  for (int l = 0; l < L; ++l) {
    const hyb_layer_io_t& io = layers[l];
    const int lt = layer_types[l];
    if (lt == HYB_SLIDING ? io.window <= 0 : io.window != 0) return HYB_ERR_INVALID_ARG;
    if (lt == HYB_FULL || lt == HYB_SLIDING) {
      if (!io.k_cache || !io.v_cache || !seen.insert(io.k_cache).second ||
          !seen.insert(io.v_cache).second)
        return HYB_ERR_INVALID_ARG;
      hyb_attn_dims_t dl = *d;
      dl.window = io.window;
      static const int64_t dummy_slot = 0;   // decode: a null slot mapping is allowed (see A7)
      st = check_append(io.k, io.v,
                        mode == HYB_MODE_DECODE && !meta->slot_mapping ? &dummy_slot
                                                                       : meta->slot_mapping,
                        T, io.k_cache, io.v_cache, &dl);
      if (st != HYB_OK) return st;
      st = mode == HYB_MODE_DECODE
               ? check_decode(io.out, io.q, io.k_cache, io.v_cache, meta->block_tables,
                              meta->seq_lens, B, meta->max_seq_len, &dl, workspace, ws_bytes)
               : check_prefill(io.out, io.q, io.k_cache, io.v_cache, meta->block_tables,
                               meta->cu_q_lens, meta->ctx_lens, B, T, meta->max_q_len, &dl);
    } else if (lt == HYB_LINEAR) {
      if (!io.state_pool || !seen.insert(io.state_pool).second) return HYB_ERR_INVALID_ARG;
      st = mode == HYB_MODE_DECODE
               ? check_linear_common(io.out, io.q, io.k, io.v, io.state_pool, io.num_state_slots,
                                     meta->state_slots, B, H, D, dt)
               : check_linear_prefill(io.out, io.q, io.k, io.v, meta->cu_q_lens, meta->ctx_lens,
                                      io.state_pool, io.num_state_slots, meta->state_slots,
                                      meta->reset, B, T, meta->max_q_len, H, D, chunk_size, dt,
                                      workspace, ws_bytes);
    } else {
      return HYB_ERR_INVALID_ARG;
    }
    if (st != HYB_OK) return st;
  }
  if (L == 0 || B == 0) return HYB_OK;
  unsigned* sw = status_word();
  if (!sw) return HYB_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  const bool trace = trace_on(s);
  if (trace) {
    g_trace.layers = 0;
    cudaEvent_t e0 = trace_event(0);
    if (!e0 || cudaEventRecord(e0, s) != cudaSuccess) return HYB_ERR_CUDA;
    std::fprintf(stderr, "hyb: dispatch %s, %d layers, batch %d, %d rows\n",
                 mode == HYB_MODE_DECODE ? "decode" : "prefill", L, B, T);
  }
  // 2) run the plan in layer order
  for (int l = 0; l < L; ++l) {
    const hyb_layer_io_t& io = layers[l];
    if (trace)
      std::fprintf(stderr, "hyb:   layer %d %s -> %s\n", l,
                   layer_types[l] == HYB_LINEAR ? "linear" : layer_types[l] == HYB_SLIDING ? "sliding" : "full",
                   layer_kernels(layer_types[l], mode, d, chunk_size));
    if (layer_types[l] == HYB_FULL || layer_types[l] == HYB_SLIDING) {
      hyb_attn_dims_t dl = *d;
      dl.window = io.window;
      if (mode == HYB_MODE_DECODE) {         // append fused into the decode launch
        // after the first layer, the kernel before this one is a layer of this dispatch,
        // which writes none of this layer's cache and none of the batch metadata
        const DecodeAppend app{io.k, io.v, meta->slot_mapping};
        st = run_decode(io.out, io.q, io.k_cache, io.v_cache, meta->block_tables, meta->seq_lens,
                        B, meta->max_seq_len, &dl, workspace, sw, s, &app, l > 0);
      } else {
        st = cuda_status(launch_kv_append(io.k, io.v, meta->slot_mapping, T, H, D, esize_of(dt),
                                          d->num_blocks, d->block_size, io.k_cache, io.v_cache,
                                          sw, s));
        if (st != HYB_OK) return st;
        st = run_prefill(io.out, io.q, io.k_cache, io.v_cache, meta->block_tables,
                         meta->cu_q_lens, meta->ctx_lens, B, T, meta->max_q_len, &dl, sw, s);
      }
    } else {
      st = mode == HYB_MODE_DECODE
               ? cuda_status(launch_linear_step(io.out, io.q, io.k, io.v, io.state_pool,
                                                io.num_state_slots, meta->state_slots, B, H, D,
                                                dt, sw, s, l > 0))
               : run_linear_prefill(io.out, io.q, io.k, io.v, meta->cu_q_lens, meta->ctx_lens,
                                    io.state_pool, io.num_state_slots, meta->state_slots,
                                    meta->reset, B, T, meta->max_q_len, H, D, chunk_size, dt,
                                    workspace, sw, s);
    }
    if (st != HYB_OK) return st;
    if (trace) {
      cudaEvent_t e = trace_event(l + 1);
      if (!e || cudaEventRecord(e, s) != cudaSuccess) return HYB_ERR_CUDA;
    }
  }
  if (trace) g_trace.layers = L;
  return HYB_OK;
}

uint64_t hyb_cache_bytes(int32_t L_full, int32_t L_linear, int32_t H, int32_t D, int64_t tokens,
                         int32_t batch, int32_t kv_elem_bytes, int32_t state_elem_bytes,
                         uint64_t* full_out, uint64_t* linear_out) {
  const uint64_t full = 2ull * (uint64_t)L_full * (uint64_t)H * (uint64_t)D * (uint64_t)tokens *
                        (uint64_t)batch * (uint64_t)kv_elem_bytes;
  const uint64_t lin = (uint64_t)L_linear * (uint64_t)H * (uint64_t)D * (uint64_t)D *
                       (uint64_t)batch * (uint64_t)state_elem_bytes;
  if (full_out) *full_out = full;
  if (linear_out) *linear_out = lin;
  return full + lin;
}

hyb_status_t hyb_device_status(uint32_t* flags, int32_t clear) {
  if (!flags) return HYB_ERR_INVALID_ARG;
  unsigned* sw = status_word();
  if (!sw) return HYB_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return HYB_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, sw, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return HYB_ERR_CUDA;
  if (clear && cudaMemset(sw, 0, sizeof(unsigned)) != cudaSuccess) return HYB_ERR_CUDA;
  if (clear && cudaDeviceSynchronize() != cudaSuccess) return HYB_ERR_CUDA;
  *flags = v;
  return v ? HYB_ERR_DEVICE_CHECK : HYB_OK;
}

const char* hyb_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda); }

const char* hyb_status_string(hyb_status_t s) {
  switch (s) {
    case HYB_OK: return "ok";
    case HYB_ERR_INVALID_ARG: return "invalid argument (nothing launched)";
    case HYB_ERR_UNSUPPORTED: return "unsupported shape or dtype (nothing launched)";
    case HYB_ERR_CUDA: return "CUDA runtime error";
    case HYB_ERR_DEVICE_CHECK: return "a device-side check failed (see hyb_device_status flags)";
  }
  return "unknown status";
}

hyb_status_t hyb_selftest_bounded_waits(uint32_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return HYB_ERR_INVALID_ARG;
  unsigned* sw = hyb::status_word();
  if (!sw) return HYB_ERR_CUDA;
  hyb::selftest_bounded_waits_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(
      (uint64_t)limit_us * 1000ull, sw);
  hyb::count_launch();
  return cuda_status(cudaGetLastError());
}

uint64_t hyb_launch_count(int32_t reset) {
  const uint64_t n = g_launches;
  if (reset) g_launches = 0;
  return n;
}

}  // extern "C"
