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
//
// Size limit: a batch with more than one split of 512 keys needs
// B x H x ceil(max_seq_len / 512) x (4 D + 8) bytes of partials; beyond 16 MiB the call
// returns HYB_ERR_UNSUPPORTED and launches nothing (at H = 32, D = 128: B x splits <= 1008).
#include <cuda_runtime.h>

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
// current, and cached. The cache assumes the device's primary context lives as long as the
// process: after cudaDeviceReset the cached address is stale.
cudaError_t scratch_address(void** addr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

hyb_status_t hyb_paged_attn_decode_noalloc(void* out, const void* q, const void* k_cache,
                                           const void* v_cache, const int32_t* block_tables,
                                           const int32_t* seq_lens, int32_t B,
                                           int32_t max_seq_len, const hyb_attn_dims_t* d,
                                           void* stream) {
  // the same argument checks as hyb_paged_attn_decode, before any CUDA call
  hyb_status_t st = hyb::check_decode_args(out, q, k_cache, v_cache, block_tables, seq_lens, B,
                                           max_seq_len, d);
  if (st != HYB_OK || B == 0) return st;
  const hyb::DecodePlan plan = hyb::plan_decode(B, d->num_heads, d->head_dim, max_seq_len,
                                                 d->window);
  if (plan.ws_bytes > kNoAllocScratchBytes) return HYB_ERR_UNSUPPORTED;   // too big: no launch
  void* scratch = nullptr;
  st = hyb::cuda_status(scratch_address(&scratch));
  if (st != HYB_OK) return st;
  unsigned* status = hyb::status_word();
  if (!status) return HYB_ERR_CUDA;
  return hyb::cuda_status(hyb::launch_paged_decode(
      out, q, k_cache, v_cache, block_tables, seq_lens, nullptr, nullptr, B, 0, d->num_heads,
      d->head_dim, d->dtype, d->num_blocks, d->max_blocks_per_seq, d->block_size, max_seq_len,
      d->scale, d->window, plan, scratch, status, (cudaStream_t)stream));
}

}  // extern "C"
