// Linear-attention decode step and the CUDA-core form of chunked prefill.
//
// Page: "推理框架适配Hybrid Model：KV Cache管理与算子调度实战", §2.1 -- each linear layer
// keeps a D x D state per head (H x D x D per request) updated per token as
// S <- S + k (outer) v with output q.S, a cost of O(D^2) per decode step; §2.3 -- the op
// takes Q, K, V and the previous state and returns the output and the new state, the
// state is zeroed at request start, accumulated in prefill and carried into decode, and
// is kept in fp32.
//
// Readings used throughout: k (outer) v = k v^T (row i = key dim, column j = value dim);
// the output reads the state after the token's own update; no feature map, normaliser,
// decay or scale.
//
// Decode step design (GB300): pure HBM traffic -- each (request, head) state is read and
// written once (2 x 64 KiB at D = 128, fp32), 0.5 flop/byte. A CTA owns 32 columns of one
// state: 8 threads x float4 cover a row, 32 rows per pass, all passes' loads issued
// before any use so each thread keeps 64 B in flight; streaming cache hints keep the
// states from evicting other data from L2. Column partial sums of q.S reduce in shared
// memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "hyb_internal.cuh"

namespace hyb {

namespace {

template <typename T>
__device__ __forceinline__ float ldf(const T* p);
template <>
__device__ __forceinline__ float ldf<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void stf(T* p, float x);
template <>
__device__ __forceinline__ void stf<float>(float* p, float x) { *p = x; }
template <>
__device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

template <int D>
struct StepShape {
  static constexpr int COLS = D < 32 ? D : 32;              // state columns per CTA
  static constexpr int TPR = COLS / 4;                      // threads per row (float4 each)
  static constexpr int THREADS = D * TPR < 256 ? D * TPR : 256;
  static constexpr int RPP = THREADS / TPR;                 // rows per pass
  static constexpr int PASSES = D / RPP;
  static_assert(PASSES * RPP == D, "shape");
};

template <typename T, int D>
__global__ void __launch_bounds__(StepShape<D>::THREADS)
linear_step_kernel(T* __restrict__ out, const T* __restrict__ q, const T* __restrict__ k,
                   const T* __restrict__ v, float* __restrict__ pool, int NS,
                   const int32_t* __restrict__ slots, int H, int early, unsigned* status) {
  using Sh = StepShape<D>;
  constexpr int COLS = Sh::COLS, TPR = Sh::TPR, RPP = Sh::RPP, PASSES = Sh::PASSES;
  __shared__ float red[RPP][COLS];

  // early (a step after another layer of the same dispatch): no kernel before it in the
  // dispatch writes anything this step reads or writes (its state, q, k, v, out, the slots), so
  // it runs while the previous kernel drains and waits for that kernel only at its end (so the
  // next kernel's wait covers every earlier kernel of the dispatch).
  if (!early) pdl_wait();
  const int cb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int slot = slots[b];
  if (slot < 0 || slot >= NS) {
    if (cb == 0 && h == 0 && threadIdx.x == 0) flag(status, HYB_DEVERR_BAD_STATE);
    return;
  }
  const int tc = threadIdx.x % TPR, rg = threadIdx.x / TPR;
  const int col = cb * COLS + tc * 4;
  const int64_t rowq = ((int64_t)b * H + h) * D;
  float* S = pool + ((int64_t)slot * H + h) * D * D;

  float4 st[PASSES];
#pragma unroll
  for (int p = 0; p < PASSES; ++p)
    st[p] = __ldcs(reinterpret_cast<const float4*>(S + (int64_t)(rg + p * RPP) * D + col));
  pdl_trigger();                           // the next kernel may launch (it waits for this one)
  const float v0 = ldf(v + rowq + col), v1 = ldf(v + rowq + col + 1);
  const float v2 = ldf(v + rowq + col + 2), v3 = ldf(v + rowq + col + 3);

  float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int i = rg + p * RPP;
    const float ki = ldf(k + rowq + i), qi = ldf(q + rowq + i);
    float4 s = st[p];
    s.x = fmaf(ki, v0, s.x);
    s.y = fmaf(ki, v1, s.y);
    s.z = fmaf(ki, v2, s.z);
    s.w = fmaf(ki, v3, s.w);
    __stcs(reinterpret_cast<float4*>(S + (int64_t)i * D + col), s);
    o0 = fmaf(qi, s.x, o0);
    o1 = fmaf(qi, s.y, o1);
    o2 = fmaf(qi, s.z, o2);
    o3 = fmaf(qi, s.w, o3);
  }
  red[rg][tc * 4 + 0] = o0;
  red[rg][tc * 4 + 1] = o1;
  red[rg][tc * 4 + 2] = o2;
  red[rg][tc * 4 + 3] = o3;
  __syncthreads();
  for (int j = threadIdx.x; j < COLS; j += Sh::THREADS) {
    float o = 0.f;
#pragma unroll 8
    for (int g = 0; g < RPP; ++g) o += red[g][j];
    stf(out + rowq + cb * COLS + j, o);
  }
  if (early) pdl_wait();
}

// 16-bit state elements for the state-precision comparison: widen exactly, round once (RNE).
template <typename S>
struct State16;
template <>
struct State16<__nv_bfloat16> {
  __device__ static float get(uint32_t w, int hi) { return hi ? bf16_hi(w) : bf16_lo(w); }
  __device__ static uint32_t pack(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&p);
  }
};
template <>
struct State16<__half> {
  __device__ static float get(uint32_t w, int hi) {
    return __half2float(__ushort_as_half((unsigned short)(hi ? w >> 16 : w & 0xffffu)));
  }
  __device__ static uint32_t pack(float lo, float hi) {
    const __half2 p = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&p);
  }
};

// 16-bit state: each thread takes 8 state columns, one 16-byte load and store per row, so
// a thread keeps as many bytes in flight as the fp32 step does with its 4 columns.
template <int D>
struct StepShape16 {
  static constexpr int COLS = D < 64 ? D : 64;              // state columns per CTA
  static constexpr int TPR = COLS / 8;                      // threads per row (8 columns each)
  static constexpr int THREADS = D * TPR < 256 ? D * TPR : 256;
  static constexpr int RPP = THREADS / TPR;                 // rows per pass
  static constexpr int PASSES = D / RPP;
  static_assert(PASSES * RPP == D && TPR >= 1, "shape");
};

template <typename T, typename S16, int D>
__global__ void __launch_bounds__(StepShape16<D>::THREADS)
linear_step_lowp_kernel(T* __restrict__ out, const T* __restrict__ q, const T* __restrict__ k,
                        const T* __restrict__ v, uint16_t* __restrict__ pool, int NS,
                        const int32_t* __restrict__ slots, int H, unsigned* status) {
  using Sh = StepShape16<D>;
  using Q = State16<S16>;
  constexpr int COLS = Sh::COLS, TPR = Sh::TPR, RPP = Sh::RPP, PASSES = Sh::PASSES;
  __shared__ float red[RPP][COLS];

  const int cb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int slot = slots[b];
  if (slot < 0 || slot >= NS) {
    if (cb == 0 && h == 0 && threadIdx.x == 0) flag(status, HYB_DEVERR_BAD_STATE);
    return;
  }
  const int tc = threadIdx.x % TPR, rg = threadIdx.x / TPR;
  const int col = cb * COLS + tc * 8;
  const int64_t rowq = ((int64_t)b * H + h) * D;
  uint16_t* S = pool + ((int64_t)slot * H + h) * D * D;

  uint4 st[PASSES];
#pragma unroll
  for (int p = 0; p < PASSES; ++p)
    st[p] = __ldcs(reinterpret_cast<const uint4*>(S + (int64_t)(rg + p * RPP) * D + col));
  float vv[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) vv[e] = ldf(v + rowq + col + e);

  float o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = 0.f;
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int i = rg + p * RPP;
    const float ki = ldf(k + rowq + i), qi = ldf(q + rowq + i);
    const uint32_t in[4] = {st[p].x, st[p].y, st[p].z, st[p].w};
    uint32_t w[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      w[c] = Q::pack(fmaf(ki, vv[2 * c], Q::get(in[c], 0)), fmaf(ki, vv[2 * c + 1], Q::get(in[c], 1)));
    __stcs(reinterpret_cast<uint4*>(S + (int64_t)i * D + col), make_uint4(w[0], w[1], w[2], w[3]));
#pragma unroll
    for (int c = 0; c < 4; ++c) {                    // the output reads the rounded state
      o[2 * c] = fmaf(qi, Q::get(w[c], 0), o[2 * c]);
      o[2 * c + 1] = fmaf(qi, Q::get(w[c], 1), o[2 * c + 1]);
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) red[rg][tc * 8 + e] = o[e];
  __syncthreads();
  for (int j = threadIdx.x; j < COLS; j += Sh::THREADS) {
    float acc = 0.f;
#pragma unroll 8
    for (int g = 0; g < RPP; ++g) acc += red[g][j];
    stf(out + rowq + cb * COLS + j, acc);
  }
}

// Chunked prefill on the CUDA cores (any D <= 128, bf16 or fp32, any chunk size): the
// token recurrence, which the chunk form equals exactly in real arithmetic. One CTA per
// (request, head), state resident in shared memory for the whole call.
template <typename T, int D>
__global__ void __launch_bounds__(256)
linear_prefill_simt_kernel(T* __restrict__ out, const T* __restrict__ q,
                           const T* __restrict__ k, const T* __restrict__ v,
                           const int32_t* __restrict__ cu, const int32_t* __restrict__ ctx,
                           float* __restrict__ pool, int NS, const int32_t* __restrict__ slots,
                           const uint8_t* __restrict__ reset, int H, int C, unsigned* status) {
  extern __shared__ float sm[];
  float* S = sm;                 // [D][D]
  float* qs = S + D * D;         // [D]
  float* ks = qs + D;
  float* vs = ks + D;
  const int h = blockIdx.x, b = blockIdx.y;
  const int slot = slots[b];
  if (slot < 0 || slot >= NS) {
    if (h == 0 && threadIdx.x == 0) flag(status, HYB_DEVERR_BAD_STATE);
    return;
  }
  if (ctx && (ctx[b] % C) != 0) {
    if (h == 0 && threadIdx.x == 0) flag(status, HYB_DEVERR_MISALIGNED);
    return;
  }
  float* Sg = pool + ((int64_t)slot * H + h) * D * D;
  const bool zero = reset && reset[b];
  for (int e = threadIdx.x; e < D * D; e += blockDim.x) S[e] = zero ? 0.f : Sg[e];
  for (int t = cu[b]; t < cu[b + 1]; ++t) {
    const int64_t row = ((int64_t)t * H + h) * D;
    __syncthreads();
    for (int i = threadIdx.x; i < D; i += blockDim.x) {
      qs[i] = ldf(q + row + i);
      ks[i] = ldf(k + row + i);
      vs[i] = ldf(v + row + i);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < D * D; e += blockDim.x) S[e] = fmaf(ks[e / D], vs[e % D], S[e]);
    __syncthreads();
    for (int j = threadIdx.x; j < D; j += blockDim.x) {
      float o = 0.f;
      for (int i = 0; i < D; ++i) o = fmaf(qs[i], S[i * D + j], o);
      stf(out + row + j, o);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < D * D; e += blockDim.x) Sg[e] = S[e];
}

template <typename T, int D>
cudaError_t step_typed(void* out, const void* q, const void* k, const void* v, float* pool,
                       int NS, const int32_t* slots, int B, int H, unsigned* status,
                       cudaStream_t s, bool early) {
  using Sh = StepShape<D>;
  dim3 grid(D / Sh::COLS, H, B);
  const cudaError_t e = launch_pdl(linear_step_kernel<T, D>, grid, dim3(Sh::THREADS), 0, s, (T*)out,
                                   (const T*)q, (const T*)k, (const T*)v, pool, NS, slots, H,
                                   early ? 1 : 0, status);
  count_launch();
  return e;
}

template <typename T, typename S16, int D>
cudaError_t step_lowp_typed(void* out, const void* q, const void* k, const void* v, void* pool,
                            int NS, const int32_t* slots, int B, int H, unsigned* status,
                            cudaStream_t s) {
  using Sh = StepShape16<D>;
  dim3 grid(D / Sh::COLS, H, B);
  linear_step_lowp_kernel<T, S16, D><<<grid, Sh::THREADS, 0, s>>>(
      (T*)out, (const T*)q, (const T*)k, (const T*)v, static_cast<uint16_t*>(pool), NS, slots, H,
      status);
  count_launch();
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t prefill_simt_typed(void* out, const void* q, const void* k, const void* v,
                               const int32_t* cu, const int32_t* ctx, float* pool, int NS,
                               const int32_t* slots, const uint8_t* reset, int B, int H, int C,
                               unsigned* status, cudaStream_t s) {
  const int smem = (D * D + 3 * D) * 4;
  cudaError_t e = set_smem((const void*)linear_prefill_simt_kernel<T, D>, smem);
  if (e != cudaSuccess) return e;
  linear_prefill_simt_kernel<T, D><<<dim3(H, B), 256, smem, s>>>(
      (T*)out, (const T*)q, (const T*)k, (const T*)v, cu, ctx, pool, NS, slots, reset, H, C,
      status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

bool linear_supported(int dtype, int D) {
  if (dtype != HYB_BF16 && dtype != HYB_F32) return false;
  return D == 16 || D == 32 || D == 64 || D == 128 || D == 256;
}

cudaError_t launch_linear_step(void* out, const void* q, const void* k, const void* v,
                               float* pool, int NS, const int32_t* slots, int B, int H, int D,
                               int dtype, unsigned* status, cudaStream_t s, bool early) {
  if (B == 0) return cudaSuccess;
#define HYB_STEP(T, DD) \
  if (D == DD) return step_typed<T, DD>(out, q, k, v, pool, NS, slots, B, H, status, s, early);
  if (dtype == HYB_BF16) {
    HYB_STEP(__nv_bfloat16, 16) HYB_STEP(__nv_bfloat16, 32) HYB_STEP(__nv_bfloat16, 64)
    HYB_STEP(__nv_bfloat16, 128) HYB_STEP(__nv_bfloat16, 256)
  } else {
    HYB_STEP(float, 16) HYB_STEP(float, 32) HYB_STEP(float, 64) HYB_STEP(float, 128)
    HYB_STEP(float, 256)
  }
#undef HYB_STEP
  return cudaErrorInvalidValue;
}

cudaError_t launch_linear_step_lowp(void* out, const void* q, const void* k, const void* v,
                                    void* pool, int state_dtype, int NS, const int32_t* slots,
                                    int B, int H, int D, int dtype, unsigned* status,
                                    cudaStream_t s) {
  if (B == 0) return cudaSuccess;
#define HYB_LSTEP(T, S16, DD)                                                              \
  if (D == DD)                                                                             \
    return step_lowp_typed<T, S16, DD>(out, q, k, v, pool, NS, slots, B, H, status, s);
#define HYB_LSTEP_D(T, S16)                                                                \
  HYB_LSTEP(T, S16, 16) HYB_LSTEP(T, S16, 32) HYB_LSTEP(T, S16, 64) HYB_LSTEP(T, S16, 128)  \
  HYB_LSTEP(T, S16, 256)
  if (dtype == HYB_BF16 && state_dtype == HYB_BF16) { HYB_LSTEP_D(__nv_bfloat16, __nv_bfloat16) }
  if (dtype == HYB_BF16 && state_dtype == HYB_F16) { HYB_LSTEP_D(__nv_bfloat16, __half) }
  if (dtype == HYB_F32 && state_dtype == HYB_BF16) { HYB_LSTEP_D(float, __nv_bfloat16) }
  if (dtype == HYB_F32 && state_dtype == HYB_F16) { HYB_LSTEP_D(float, __half) }
#undef HYB_LSTEP_D
#undef HYB_LSTEP
  return cudaErrorInvalidValue;
}

cudaError_t launch_linear_prefill_simt(void* out, const void* q, const void* k, const void* v,
                                       const int32_t* cu, const int32_t* ctx, float* pool,
                                       int NS, const int32_t* slots, const uint8_t* reset, int B,
                                       int H, int D, int C, int dtype, unsigned* status,
                                       cudaStream_t s) {
  if (B == 0) return cudaSuccess;
#define HYB_PF(T, DD)                                                                      \
  if (D == DD)                                                                             \
    return prefill_simt_typed<T, DD>(out, q, k, v, cu, ctx, pool, NS, slots, reset, B, H, C, \
                                     status, s);
  if (dtype == HYB_BF16) {
    HYB_PF(__nv_bfloat16, 16) HYB_PF(__nv_bfloat16, 32) HYB_PF(__nv_bfloat16, 64)
    HYB_PF(__nv_bfloat16, 128)
  } else {
    HYB_PF(float, 16) HYB_PF(float, 32) HYB_PF(float, 64) HYB_PF(float, 128)
  }
#undef HYB_PF
  return cudaErrorInvalidValue;
}

}  // namespace hyb
