// Chunked linear-attention prefill on the tensor cores (tcgen05 + TMEM + TMA), bf16 q/k/v,
// D = 128, chunk C = 64, fp32 state.
//
// Page: "推理框架适配Hybrid Model：KV Cache管理与算子调度实战", §2.1 (state update
// S <- S + k (outer) v, output q.S), §2.3 (state zeroed at request start, accumulated in
// prefill, kept in fp32) and §2.4 (chunks carry the state; chunk boundaries aligned).
// Per chunk c of a (request, head), with S the fp32 state at the chunk start:
//     O_c = Q_c S + tril(Q_c K_c^T) V_c        S <- S + K_c^T V_c
//
// GB300 design. One CTA per (request, head) walks its chunks in order (the state chain is
// sequential); 256 chains of the 8 x 8192-token prompt fill the 152 SMs in under two
// waves. Q/K/V chunks stream through a 3-stage TMA ring (SW128 tiles, one mbarrier per
// stage). The state lives in TMEM for the whole call and is accumulated in place by the
// tensor core. Four MMA groups per chunk (M x N x K):
//   (a) P    = Q_c K_c^T          64 x 64 x 128   A = Q (K-major), B = K (K-major)
//   (b) O^T  = S^T Q_c^T          128 x 64 x 128  A = S^T (MN-major, bf16 hi and lo parts),
//                                                 B = Q (K-major); hi + lo keeps ~16 bits
//   (d) S   += K_c^T V_c          128 x 128 x 64  A = K^T (MN-major), B = V (MN-major)
//   (c) O^T += V_c^T tril(P)^T    128 x 64 x 64   A = V^T (MN-major), B = tril(P) (K-major)
// Eight conversion warps move TMEM -> registers -> shared memory: the causal mask and bf16
// rounding of P, the hi/lo split of S for the next chunk's (b), and O^T -> global (one
// column of O per thread, so stores of a warp are 64 contiguous bytes). One warp issues
// TMA and MMA (lane 0) and zeroes the K/V rows past the end of a request's last chunk.
// Output is computed transposed (M = value dim) so every MMA but (a) uses M = 128.
#include <cuda_bf16.h>

#include "tc.cuh"

namespace hyb {
namespace {

constexpr int kC = 64, kD = 128;
constexpr int kNST = 3;                      // Q/K/V ring stages
constexpr int kSub = 64 * 128;               // bytes of one [64 rows][64 cols] SW128 sub-tile
constexpr int kTile = 2 * kSub;              // [64][128] bf16 tile
constexpr int kStage = 3 * kTile;            // Q, K, V
constexpr int kOffS = kNST * kStage;         // S^T hi / lo (each [128 k-rows][128], MN-major)
constexpr int kSTile = 128 * 128 * 2;
constexpr int kOffP = kOffS + 2 * kSTile;    // tril(P) [64][64] K-major
constexpr int kOffBar = kOffP + kSub;
constexpr int kSmem = kOffBar + 256 + 1024;  // + slack for 1024-byte alignment
constexpr int kNCW = 8;                      // conversion warps
constexpr int kThreads = (kNCW + 1) * 32;
constexpr uint32_t kTmemCols = 256;          // S [0,128) | O^T [128,192) | P [192,256)
constexpr uint32_t kColS = 0, kColO = 128, kColP = 192;

constexpr uint32_t kIdescA = idesc_bf16(64, 64, 0, 0);
constexpr uint32_t kIdescB = idesc_bf16(128, 64, 1, 0);
constexpr uint32_t kIdescD = idesc_bf16(128, 128, 1, 1);
constexpr uint32_t kIdescC = idesc_bf16(128, 64, 1, 0);

struct Bars {
  uint64_t full[kNST], empty[kNST];
  uint64_t p_ready, p_written, s_ready, s_written, o_ready, o_read, drain;
};

__global__ void __launch_bounds__(kThreads, 1)
linear_prefill_tc_kernel(const __grid_constant__ CUtensorMap tq,
                         const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv, __nv_bfloat16* __restrict__ out,
                         const int32_t* __restrict__ cu, const int32_t* __restrict__ ctx,
                         float* __restrict__ pool, int NS, const int32_t* __restrict__ slots,
                         const uint8_t* __restrict__ reset, int H, unsigned* status) {
  const int h = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = cu[b], n = cu[b + 1] - t0;
  const int slot = slots[b];
  if (slot < 0 || slot >= NS) {
    if (h == 0 && tid == 0) flag(status, HYB_DEVERR_BAD_STATE);
    return;
  }
  if (ctx && (ctx[b] % kC) != 0) {
    if (h == 0 && tid == 0) flag(status, HYB_DEVERR_MISALIGNED);
    return;
  }
  float* Sg = pool + ((int64_t)slot * H + h) * kD * kD;
  const bool zero_start = reset && reset[b];
  if (n <= 0) {                              // no rows: only a reset has an effect
    if (zero_start)
      for (int e = tid; e < kD * kD / 4; e += kThreads)
        reinterpret_cast<float4*>(Sg)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int nch = (n + kC - 1) / kC;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(sm + kOffBar);
  __shared__ uint32_t tmem_base;

  if (warp == kNCW) {
    if (lane == 0) {
      for (int s = 0; s < kNST; ++s) {
        mbar_init(&bars->full[s], 1);
        mbar_init(&bars->empty[s], 1);
      }
      mbar_init(&bars->p_ready, 1);
      mbar_init(&bars->s_ready, 1);
      mbar_init(&bars->o_ready, 1);
      mbar_init(&bars->p_written, kNCW * 32);
      mbar_init(&bars->s_written, kNCW * 32);
      mbar_init(&bars->o_read, kNCW * 32);
      mbar_init(&bars->drain, 1);
      fence_mbar_init();
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
    }
    __syncwarp();
    tmem_alloc(&tmem_base, kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  uint8_t* const s_hi = sm + kOffS;
  uint8_t* const s_lo = s_hi + kSTile;
  uint8_t* const p_tile = sm + kOffP;

  if (warp == kNCW) {
    // ------------------------------------------------------------ TMA + MMA warp
    bool ok = true;
    int issued = 0, consumed = 0;            // chunks whose loads were issued / waited for
    auto load = [&](int c) {                 // lane 0
      const int st = c % kNST;
      uint8_t* q = sm + st * kStage;
      uint64_t* bar = &bars->full[st];
      mbar_expect_tx(bar, kStage);
      const int z = t0 + c * kC;
      for (int sb = 0; sb < 2; ++sb) {
        tma_load_3d(q + sb * kSub, &tq, sb * 64, h, z, bar);
        tma_load_3d(q + kTile + sb * kSub, &tk, sb * 64, h, z, bar);
        tma_load_3d(q + 2 * kTile + sb * kSub, &tv, sb * 64, h, z, bar);
      }
    };
    if (lane == 0)
      for (int c = 0; c < min(kNST, nch); ++c) load(c);
    issued = min(kNST, nch);
    for (int c = 0; c < nch && ok; ++c) {
      const int st = c % kNST;
      uint8_t* qs = sm + st * kStage;
      uint8_t* ks = qs + kTile;
      uint8_t* vs = ks + kTile;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->full[st], (c / kNST) & 1));
      if (!ok) break;
      consumed = c + 1;
      const int nvalid = min(kC, n - c * kC);
      if (nvalid < kC) {                     // rows past the request: K and V rows := 0
        for (int e = lane; e < (kC - nvalid) * 2 * 8; e += 32) {
          const int r = nvalid + e / 16, sb = (e / 8) & 1, ch = e & 7;
          const uint4 z4 = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(ks + sb * kSub + r * 128 + ch * 16) = z4;
          *reinterpret_cast<uint4*>(vs + sb * kSub + r * 128 + ch * 16) = z4;
        }
        fence_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        tc_fence_after();
        const uint32_t qa = smem_u32(qs), ka = smem_u32(ks);
#pragma unroll
        for (int k = 0; k < 8; ++k) {        // (a) P = Q K^T
          const uint32_t off = (k >> 2) * kSub + (k & 3) * 32;
          tc_mma(tmem + kColP, sw128_desc(qa + off, 16, 1024), sw128_desc(ka + off, 16, 1024),
                 kIdescA, k > 0);
        }
        tc_commit(&bars->p_ready);
      }
      // refill the stage the previous chunk used, once its MMAs are done
      if (c >= 1 && c - 1 + kNST < nch) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->empty[(c - 1) % kNST], ((c - 1) / kNST) & 1));
        if (!ok) break;
        if (lane == 0) load(c - 1 + kNST);
        issued = c - 1 + kNST + 1;
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_written, c & 1));
      if (ok && c > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_read, (c - 1) & 1));
      if (!ok) break;
      if (lane == 0) {
        tc_fence_after();
        const uint32_t qa = smem_u32(qs), ka = smem_u32(ks), va = smem_u32(vs);
        const uint32_t ha = smem_u32(s_hi), la = smem_u32(s_lo);
#pragma unroll
        for (int part = 0; part < 2; ++part) {   // (b) O^T = S^T Q^T, hi then lo
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t a = (part ? la : ha) + k * 2048;
            const uint32_t boff = (k >> 2) * kSub + (k & 3) * 32;
            tc_mma(tmem + kColO, sw128_desc(a, 16384, 1024), sw128_desc(qa + boff, 16, 1024),
                   kIdescB, (part | k) != 0);
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)              // (d) S += K^T V
          tc_mma(tmem + kColS, sw128_desc(ka + k * 2048, kSub, 1024),
                 sw128_desc(va + k * 2048, kSub, 1024), kIdescD, 1);
        tc_commit(&bars->s_ready);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_written, c & 1));
      if (!ok) break;
      if (lane == 0) {
        tc_fence_after();
        const uint32_t va = smem_u32(vs), pa = smem_u32(p_tile);
#pragma unroll
        for (int k = 0; k < 4; ++k)              // (c) O^T += V^T tril(P)^T
          tc_mma(tmem + kColO, sw128_desc(va + k * 2048, kSub, 1024),
                 sw128_desc(pa + k * 32, 16, 1024), kIdescC, 1);
        tc_commit(&bars->o_ready);
        tc_commit(&bars->empty[st]);
      }
    }
    if (!ok) {
      // A wait expired: report it, then let every issued MMA and TMA load land (bounded)
      // before the CTA releases its shared memory and TMEM.
      if (lane == 0) {
        flag(status, HYB_DEVERR_TIMEOUT);
        tc_commit(&bars->drain);
        mbar_wait(&bars->drain, 0, 100000000ull);
        for (int cc = consumed; cc < issued; ++cc)
          mbar_wait(&bars->full[cc % kNST], (cc / kNST) & 1, 100000000ull);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ conversion warps
    const int quarter = warp & 3, hf = warp >> 2;
    const int row = quarter * 32 + lane;                 // TMEM lane of this thread
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    bool ok = true;
    // initial state -> TMEM (fp32) and S^T hi/lo operands
    auto put_state = [&](const float* v, int j0) {       // 32 values, columns j0..j0+31
      const int mb = j0 >> 6;                            // MN block of the operand
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t hi4[4], lo4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = v[ch * 8 + 2 * e], x1 = v[ch * 8 + 2 * e + 1];
          const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
          hi4[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
          lo4[e] = pack_bf16(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
        }
        const int c16 = ((j0 & 63) >> 3) + ch;
        const uint32_t off = mb * 16384 + (row >> 3) * 1024 + sw128_off(row & 7, c16);
        *reinterpret_cast<uint4*>(s_hi + off) = make_uint4(hi4[0], hi4[1], hi4[2], hi4[3]);
        *reinterpret_cast<uint4*>(s_lo + off) = make_uint4(lo4[0], lo4[1], lo4[2], lo4[3]);
      }
    };
    {
      float v[32];
      for (int part = 0; part < 2; ++part) {
        const int j0 = hf * 64 + part * 32;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          float4 x = zero_start ? make_float4(0.f, 0.f, 0.f, 0.f)
                                : *reinterpret_cast<const float4*>(Sg + (int64_t)row * kD + j0 + e);
          v[e] = x.x; v[e + 1] = x.y; v[e + 2] = x.z; v[e + 3] = x.w;
        }
        tmem_st32(tl + kColS + j0, v);
        put_state(v, j0);
      }
      tmem_st_wait();
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->s_written);
    }
    for (int c = 0; c < nch && ok; ++c) {
      const int nvalid = min(kC, n - c * kC);
      float v[32];
      // ---- tril(P) -> shared (K-major [t][t'])
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_ready, c & 1));
      if (!ok) break;
      tc_fence_after();
      tmem_ld32(tl + kColP + hf * 32, v);
      tmem_ld_wait();
      if (lane < 16) {
        const int t = quarter * 16 + lane;               // M = 64 layout: lanes 0..15 of each quarter
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tp = hf * 32 + ch * 8 + 2 * e;
            w[e] = pack_bf16(tp <= t ? v[ch * 8 + 2 * e] : 0.f, tp + 1 <= t ? v[ch * 8 + 2 * e + 1] : 0.f);
          }
          *reinterpret_cast<uint4*>(p_tile + sw128_off(t, hf * 4 + ch)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_written);
      // ---- state: next chunk's S^T hi/lo operands, or the final state to global
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_ready, c & 1));
      if (!ok) break;
      tc_fence_after();
      const bool last = c == nch - 1;
      for (int part = 0; part < 2; ++part) {
        const int j0 = hf * 64 + part * 32;
        tmem_ld32(tl + kColS + j0, v);
        tmem_ld_wait();
        if (last) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(Sg + (int64_t)row * kD + j0 + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        } else {
          put_state(v, j0);
        }
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->s_written);
      // ---- O^T -> global: this thread owns value dim j = row, tokens hf*32 .. hf*32+31
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_ready, c & 1));
      if (!ok) break;
      tc_fence_after();
      tmem_ld32(tl + kColO + hf * 32, v);
      tmem_ld_wait();
      __nv_bfloat16* o = out + ((int64_t)(t0 + c * kC) * H + h) * kD + row;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int t = hf * 32 + e;
        if (t < nvalid) o[(int64_t)t * H * kD] = __float2bfloat16_rn(v[e]);
      }
      tc_fence_before();
      mbar_arrive(&bars->o_read);
    }
    if (!ok && lane == 0) flag(status, HYB_DEVERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kNCW) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool linear_prefill_tc_supported(int dtype, int D, int C) {
  return dtype == HYB_BF16 && D == kD && C == kC;
}

cudaError_t launch_linear_prefill_tc(void* out, const void* q, const void* k, const void* v,
                                     const int32_t* cu, const int32_t* ctx, float* pool, int NS,
                                     const int32_t* slots, const uint8_t* reset, int B, int T,
                                     int max_len, int H, int C, unsigned* status,
                                     cudaStream_t s) {
  (void)max_len;
  (void)C;
  if (B == 0 || T == 0) {
    if (B == 0) return cudaSuccess;
  }
  CUtensorMap mq, mk, mv;
  const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)H, (uint64_t)(T > 0 ? T : 1)};
  const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)H * kD * 2};
  const uint32_t box[3] = {64, 1, (uint32_t)kC};
  if (!encode_tmap_bf16(&mq, q, 3, dims, strides, box) ||
      !encode_tmap_bf16(&mk, k, 3, dims, strides, box) ||
      !encode_tmap_bf16(&mv, v, 3, dims, strides, box))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem((const void*)linear_prefill_tc_kernel, kSmem);
  if (e != cudaSuccess) return e;
  linear_prefill_tc_kernel<<<dim3(H, B), kThreads, kSmem, s>>>(
      mq, mk, mv, static_cast<__nv_bfloat16*>(out), cu, ctx, pool, NS, slots, reset, H, status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace hyb
