// Internal declarations shared by the libhyb.so translation units (not part of the ABI).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/hyb.h"

namespace hyb {

// Kernels walk the cache in 16-token sub-tiles (the block size of [KV §2.1]); a block of
// bs tokens (a power of two from 16 to 256) is bs / 16 consecutive sub-tiles.
constexpr int kBlockSize = 16;
constexpr bool block_size_ok(int bs) { return bs >= 16 && bs <= 256 && (bs & (bs - 1)) == 0; }
inline int log2_int(int x) { int r = 0; while ((1 << r) < x) ++r; return r; }

// ------------------------------------------------------------------ host side
void count_launch();                       // per-thread launch counter (hyb_launch_count)
unsigned* status_word();                   // this device's status word (nullptr on error)
int num_sms();                             // SMs of the current device (cached)
cudaError_t set_smem(const void* fn, int bytes);   // opt-in dynamic shared memory, once
// HYB_OK for cudaSuccess; otherwise records e for hyb_last_cuda_error and returns HYB_ERR_CUDA
hyb_status_t cuda_status(cudaError_t e);
// argument checks shared by the entry points (no CUDA call, no launch)
hyb_status_t check_dims(const hyb_attn_dims_t* d);
// every decode check except the workspace's (B == 0 returns HYB_OK before the pointer checks)
hyb_status_t check_decode_args(const void* out, const void* q, const void* kc, const void* vc,
                               const int32_t* bt, const int32_t* seq_lens, int B, int max_seq_len,
                               const hyb_attn_dims_t* d);

// Programmatic dependent launch for the short kernels of a decode step: a kernel launched
// this way may be scheduled while the previous kernel on the stream drains. It calls
// pdl_wait() before it reads anything (so stream order holds for every input) and
// pdl_trigger() once its own main work is done, so the next launch overlaps its tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// kernel launchers (each returns the launch's cudaError_t)
cudaError_t launch_slot_mapping(int64_t* slot, const int32_t* bt, const int32_t* cu,
                                const int32_t* ctx, int B, int T, int MB, int NB, int bs,
                                unsigned* status, cudaStream_t s);
cudaError_t launch_kv_append(const void* k, const void* v, const int64_t* slot, int T, int H,
                             int D, int esize, int NB, int bs, void* kc, void* vc,
                             unsigned* status, cudaStream_t s);

struct DecodePlan {
  int blocks_per_split;   // KV blocks handled by one CTA
  int max_splits;         // grid.x
  size_t ws_bytes;        // workspace needed (0 if max_splits == 1)
};
// window > 0: each row attends to at most `window` keys (sliding window)
DecodePlan plan_decode(int B, int H, int D, int max_seq_len, int window);
bool decode_supported(int dtype, int D);
// decode mode (cu == nullptr): row r < R is request r and attends to seq_lens[r] keys.
// prefill mode (cu != nullptr): R = B requests; query j < max_q of request b is packed row
// cu[b] + j and attends to ctx[b] + j + 1 keys (no split-K; no workspace).
// window > 0 keeps the last `window` of those keys.
// append (decode mode only, may be null): this step's k/v rows [R][H][D] go to the cache
// at slot[r] (-1: none) inside the decode launch, and the attention sees them; equal to a
// KV append with the same slots followed by the decode, for slot[r] = -1 or the slot of
// position seq_lens[r] - 1.
// early (decode mode): no earlier kernel that may still be running writes anything this call
// reads (its q, new row, cache, block table, lengths or slot mapping; true for every decode
// of a dispatch after its first layer); the kernel then streams its whole K/V range before
// waiting for the previous kernel, and waits before its first write of the split workspace
// or the output.
struct DecodeAppend {
  const void* k;
  const void* v;
  const int64_t* slot;
};
cudaError_t launch_paged_decode(void* out, const void* q, const void* kc, const void* vc,
                                const int32_t* bt, const int32_t* seq_lens, const int32_t* cu,
                                const int32_t* ctx, int R, int max_q, int H, int D, int dtype,
                                int NB, int MB, int bs, int max_len, float scale, int window,
                                const DecodePlan& plan, void* ws, unsigned* status,
                                cudaStream_t s, const DecodeAppend* app = nullptr,
                                bool early = false);

bool linear_supported(int dtype, int D);
// 16-bit state pool (state_dtype HYB_BF16 or HYB_F16), same shapes as launch_linear_step
cudaError_t launch_linear_step_lowp(void* out, const void* q, const void* k, const void* v,
                                    void* pool, int state_dtype, int NS, const int32_t* slots,
                                    int B, int H, int D, int dtype, unsigned* status,
                                    cudaStream_t s);
// early: as for the decode (no earlier kernel still running writes this pool, the slots or
// q/k/v); the step then waits for the previous kernel only at its end
cudaError_t launch_linear_step(void* out, const void* q, const void* k, const void* v,
                               float* pool, int NS, const int32_t* slots, int B, int H, int D,
                               int dtype, unsigned* status, cudaStream_t s, bool early = false);
cudaError_t launch_linear_prefill_simt(void* out, const void* q, const void* k, const void* v,
                                       const int32_t* cu, const int32_t* ctx, float* pool,
                                       int NS, const int32_t* slots, const uint8_t* reset, int B,
                                       int H, int D, int C, int dtype, unsigned* status,
                                       cudaStream_t s);
bool linear_prefill_tc_supported(int dtype, int D, int C);
// Handoff workspace of the tensor-core chunked prefill: a per-call epoch and one flag per CTA
// (at most kLinMaxCtas CTAs), 64-bit words.
constexpr int kLinMaxCtas = 256;
constexpr size_t kLinPrefillWsBytes = 8 * (1 + kLinMaxCtas);
cudaError_t launch_linear_prefill_tc(void* out, const void* q, const void* k, const void* v,
                                     const int32_t* cu, const int32_t* ctx, float* pool, int NS,
                                     const int32_t* slots, const uint8_t* reset, int B, int T,
                                     int max_len, int H, int C, void* ws, unsigned* status,
                                     cudaStream_t s);
bool prefill_tc_supported(int dtype, int D);
cudaError_t launch_prefill_tc(void* out, const void* q, const void* kc, const void* vc,
                              const int32_t* bt, const int32_t* cu, const int32_t* ctx, int B,
                              int T, int max_q_len, int H, int NB, int MB, int bs, float scale,
                              int window, unsigned* status, cudaStream_t s);

}  // namespace hyb

// ------------------------------------------------------------------ device side
#ifdef __CUDACC__
namespace hyb {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void flag(unsigned* st, unsigned bit) {
  if (st) atomicOr(st, bit);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 2^x with the hardware approximation (PTX ex2.approx.ftz.f32); 2^-inf = +0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- mbarrier (CTA scope)
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Waits for the phase with the given parity to complete; gives up after ~`limit_ns`
// nanoseconds and returns false (callers set HYB_DEVERR_TIMEOUT and unwind).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// ---- bulk copies (TMA engine, non-tensor form): global -> shared, completes on `bar`
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace hyb
#endif
