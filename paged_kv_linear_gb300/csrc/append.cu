// Slot mapping and KV append into the paged cache.
//
// Page: "推理框架适配Hybrid Model：KV Cache管理与算子调度实战", §2.1 -- every token's key
// and value vectors are kept; the cache is cut into blocks of a fixed number of
// tokens (16 there; 32 on the vLLM/SGLang page) allocated on demand and reached through a
// per-request page table. bs below is that block size.
//
// Both kernels are pure integer addressing plus 16-byte copies: they are bound by
// the bytes they move (T*H*D*esize read and written for K and for V).
#include "hyb_internal.cuh"

namespace hyb {

// One thread per packed row: slot = block_tables[b][p/bs]*bs + p%bs at absolute
// position p = ctx_lens[b] + (t - cu[b]). grid = (B, y): CTAs (b, y) stride over b's rows.
__global__ void slot_mapping_kernel(int64_t* __restrict__ slot, const int32_t* __restrict__ bt,
                                    const int32_t* __restrict__ cu,
                                    const int32_t* __restrict__ ctx, int MB, int NB, int bs,
                                    unsigned* status) {
  pdl_wait();
  const int b = blockIdx.x;
  const int t0 = cu[b], t1 = cu[b + 1];
  const int64_t p0 = ctx ? ctx[b] : 0;
  for (int t = t0 + blockIdx.y * blockDim.x + threadIdx.x; t < t1;
       t += gridDim.y * blockDim.x) {
    const int64_t p = p0 + (t - t0);
    const int64_t logical = p / bs;
    int64_t s = -1;
    if (logical >= MB) {
      flag(status, HYB_DEVERR_BAD_BLOCK);
    } else {
      const int32_t blk = bt[(int64_t)b * MB + logical];
      if (blk >= NB) flag(status, HYB_DEVERR_BAD_BLOCK);
      else if (blk >= 0) s = (int64_t)blk * bs + p % bs;
    }
    slot[t] = s;
  }
  pdl_trigger();
}

cudaError_t launch_slot_mapping(int64_t* slot, const int32_t* bt, const int32_t* cu,
                                const int32_t* ctx, int B, int T, int MB, int NB, int bs,
                                unsigned* status, cudaStream_t s) {
  if (B == 0 || T == 0) return cudaSuccess;
  const int per_req = (T + B - 1) / B;
  dim3 grid(B, (unsigned)std::min(64, std::max(1, (per_req + 255) / 256)));
  const cudaError_t e =
      launch_pdl(slot_mapping_kernel, grid, dim3(256), 0, s, slot, bt, cu, ctx, MB, NB, bs, status);
  count_launch();
  return e;
}

// One thread per 16-byte vector of a (token, head) row, for K and V together.
// vpr = D*esize/16 vectors per row. Rows with slot -1 are skipped; a slot beyond the
// pool is flagged and skipped.
__global__ void kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                 const int64_t* __restrict__ slot, int64_t total, int H, int vpr,
                                 int bs, int64_t n_slots, uint4* __restrict__ kc,
                                 uint4* __restrict__ vc, unsigned* status) {
  pdl_wait();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / vpr;           // t*H + h
    const int c = (int)(i - row * vpr);
    const int64_t t = row / H;
    const int h = (int)(row - t * H);
    const int64_t s = slot[t];
    if (s < 0) continue;
    if (s >= n_slots) {
      flag(status, HYB_DEVERR_BAD_SLOT);
      continue;
    }
    const int64_t blk = s / bs, off = s - blk * bs;
    const int64_t dst = ((blk * H + h) * bs + off) * vpr + c;
    kc[dst] = k[i];
    vc[dst] = v[i];
  }
  pdl_trigger();
}

cudaError_t launch_kv_append(const void* k, const void* v, const int64_t* slot, int T, int H,
                             int D, int esize, int NB, int bs, void* kc, void* vc,
                             unsigned* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int vpr = D * esize / 16;
  const int64_t total = (int64_t)T * H * vpr;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms() * 16;
  if (blocks > cap) blocks = cap;
  const cudaError_t e = launch_pdl(
      kv_append_kernel, dim3((unsigned)blocks), dim3(threads), 0, s, static_cast<const uint4*>(k),
      static_cast<const uint4*>(v), slot, total, H, vpr, bs, (int64_t)NB * bs,
      static_cast<uint4*>(kc), static_cast<uint4*>(vc), status);
  count_launch();
  return e;
}

}  // namespace hyb
