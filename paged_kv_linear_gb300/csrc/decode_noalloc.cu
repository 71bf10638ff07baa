// Paged decode attention for callers that cannot allocate device memory.
//
// hyb_paged_attn_decode needs a caller-provided workspace for its split-K partial
// softmax states. Some callers have no way to provide one: a serving runtime whose
// device memory is entirely carved up by its own planner and that only hands an op its
// input and output buffers (an inference-server plugin interface, for example), or a
// latency-critical loop that must not call cudaMalloc because it synchronises the whole
// device. This entry point keeps those partials in a fixed array of device memory that
// belongs to the library itself, so the call allocates nothing.
//
// The array is file-scope __device__ storage: every GPU that loads the library holds
// kNoAllocScratchBytes of it until the process exits. All calls on a device share it and
// it keeps whatever the previous call left there. Nothing in it has to start at zero:
// each split writes its partial (m, l, acc) in full before the merge reads it. Calls
// whose kernels overlap on the GPU (two streams, or two host threads) race on the array;
// issue them on one stream, one after another.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "hyb_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;   // 16 MiB per device

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
constexpr int kMaxDev = 64;
void* g_scratch_addr[kMaxDev] = {};

// Device address of this device's scratch array. In host code the array's name is only a
// host-side stand-in, so the real address is looked up once per device, with that device
// current, and cached.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

inline bool aligned(const void* p, unsigned a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace

extern "C" {

hyb_status_t hyb_paged_attn_decode_noalloc(void* out, const void* q, const void* k_cache,
                                           const void* v_cache, const int32_t* block_tables,
                                           const int32_t* seq_lens, int32_t B,
                                           int32_t max_seq_len, const hyb_attn_dims_t* d,
                                           void* stream) {
  if (!d || B < 0 || max_seq_len < 0) return HYB_ERR_INVALID_ARG;
  if (d->num_heads <= 0 || d->head_dim <= 0 || d->num_blocks <= 0 || d->max_blocks_per_seq <= 0)
    return HYB_ERR_INVALID_ARG;
  if (d->dtype != HYB_BF16 && d->dtype != HYB_F32) return HYB_ERR_INVALID_ARG;
  if (d->window < 0 || !std::isfinite(d->scale)) return HYB_ERR_INVALID_ARG;
  if (!hyb::block_size_ok(d->block_size) || d->num_heads > 65535 || max_seq_len > (1 << 24) ||
      !hyb::decode_supported(d->dtype, d->head_dim) ||
      (int64_t)d->num_blocks * d->num_heads * d->block_size > INT32_MAX)
    return HYB_ERR_UNSUPPORTED;
  if ((int64_t)max_seq_len > (int64_t)d->max_blocks_per_seq * d->block_size)
    return HYB_ERR_INVALID_ARG;
  if (B == 0) return HYB_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return HYB_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4))
    return HYB_ERR_INVALID_ARG;
  const hyb::DecodePlan plan = hyb::plan_decode(B, d->num_heads, d->head_dim, max_seq_len,
                                                 d->window);
  if (plan.ws_bytes > kNoAllocScratchBytes) return HYB_ERR_UNSUPPORTED;   // too big: no launch
  void* scratch = scratch_address();
  unsigned* status = hyb::status_word();
  if (!scratch || !status) return HYB_ERR_CUDA;
  const cudaError_t e = hyb::launch_paged_decode(
      out, q, k_cache, v_cache, block_tables, seq_lens, nullptr, nullptr, B, 0, d->num_heads,
      d->head_dim, d->dtype, d->num_blocks, d->max_blocks_per_seq, d->block_size, max_seq_len,
      d->scale, d->window, plan, scratch, status, (cudaStream_t)stream);
  return e == cudaSuccess ? HYB_OK : HYB_ERR_CUDA;
}

}  // extern "C"
