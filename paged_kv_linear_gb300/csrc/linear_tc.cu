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
// sequential). Warp roles: one TMA warp streams Q/K/V chunks through a 3-stage ring (SW128
// tiles, one mbarrier per stage); one MMA warp issues the tensor-core work; eight
// conversion warps move TMEM -> registers -> shared/global memory. The state lives in TMEM
// for the whole call and is accumulated in place. Per chunk (M x N x K), in issue order:
//   (d) S   += K_c^T V_c          128 x 128 x 64  A = K^T (MN-major), B = V (MN-major)
//   (b) O^T  = S^T Q_c^T          128 x 64 x 128  A = S^T of the previous chunk end, rounded
//                                                 to bf16 (the fp32 state stays in TMEM), B = Q
//   (a) P    = Q_c K_c^T          64 x 64 x 128   A = Q (K-major), B = K (K-major)
//   (c) O^T += V_c^T tril(P)^T    128 x 64 x 64   A = V^T (MN-major), B = tril(P) (K-major)
// The chain that limits a request is (d) -> read S from TMEM -> next (d): the conversion
// warps release the state as soon as they hold it in registers ("S read"), and write its
// bf16 copy for (b) only once (b) has consumed the previous one ("S written"); (c) of a
// chunk is issued after (a) of the next, so no state update waits for P's conversion. O^T and P are
// double-buffered (TMEM and shared memory) and every handshake barrier exists once per
// buffer parity, so none can run two phases ahead of its waiter. Output is computed
// transposed (M = value dim) so all MMAs but (a) use M = 128. Four conversion warps carry
// the state and P; the other four only move outputs: they write each output chunk into a
// shared staging tile (two buffers) that one thread stores with TMA (a request's last,
// partial chunk is stored directly, so no row of the next request is touched).
#include <cuda_bf16.h>

#include "tc.cuh"

namespace hyb {
namespace {

constexpr int kC = 64, kD = 128;
constexpr int kNST = 3;                      // Q/K/V ring stages
constexpr int kSub = 64 * 128;               // bytes of one [64 rows][64 cols] SW128 sub-tile
constexpr int kTile = 2 * kSub;              // [64][128] bf16 tile
constexpr int kStage = 3 * kTile;            // Q, K, V
constexpr int kOffS = kNST * kStage;         // S^T as bf16 ([128 k-rows][128], MN-major)
constexpr int kSTile = 128 * 128 * 2;
constexpr int kOffP = kOffS + kSTile;        // tril(P) [64][64] K-major, two buffers
constexpr int kOffO = kOffP + 2 * kSub;      // output staging [64 tokens][128] bf16, two buffers
constexpr int kOffBar = kOffO + 2 * kTile;
constexpr int kSmem = kOffBar + 256 + 1024;  // + slack for 1024-byte alignment
constexpr int kNCW = 8;                      // conversion warps
constexpr int kWarpTma = kNCW, kWarpMma = kNCW + 1;
constexpr int kThreads = (kNCW + 2) * 32;
constexpr uint32_t kTmemCols = 512;          // S [0,128) | O^T x2 [128,256) | P x2 [256,384)
constexpr uint32_t kColS = 0, kColO = 128, kColP = 256;

constexpr uint32_t kIdescA = idesc_bf16(64, 64, 0, 0);
constexpr uint32_t kIdescB = idesc_bf16(128, 64, 1, 0);
constexpr uint32_t kIdescD = idesc_bf16(128, 128, 1, 1);
constexpr uint32_t kIdescC = idesc_bf16(128, 64, 1, 0);

struct Bars {
  uint64_t full[kNST], empty[kNST];
  uint64_t s_ready, s_read, b_done, s_written, drain;
  uint64_t p_ready[2], p_written[2], o_ready[2], o_free[2];   // one per buffer parity
  uint64_t o_staged[2], o_stage_free[2];
};

__global__ void __launch_bounds__(kThreads, 1)
linear_prefill_tc_kernel(const __grid_constant__ CUtensorMap tq,
                         const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv,
                         const __grid_constant__ CUtensorMap to, __nv_bfloat16* __restrict__ out,
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

  if (warp == kWarpMma) {
    if (lane == 0) {
      for (int s = 0; s < kNST; ++s) {
        mbar_init(&bars->full[s], 1);
        mbar_init(&bars->empty[s], 1);
      }
      mbar_init(&bars->s_ready, 1);
      mbar_init(&bars->b_done, 1);
      mbar_init(&bars->s_read, 128);               // state warps (0-3)
      mbar_init(&bars->s_written, 128);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&bars->p_ready[i], 1);
        mbar_init(&bars->p_written[i], 128);           // state warps
        mbar_init(&bars->o_ready[i], 1);
        mbar_init(&bars->o_free[i], 128);              // output warps (4-7)
        mbar_init(&bars->o_staged[i], 128);
        mbar_init(&bars->o_stage_free[i], 1);
      }
      mbar_init(&bars->drain, 1);
      fence_mbar_init();
    }
    __syncwarp();
    tmem_alloc(&tmem_base, kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  uint8_t* const s_hi = sm + kOffS;
  uint8_t* const p_tile = sm + kOffP;
  uint8_t* const o_stage = sm + kOffO;

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA warp
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
    }
    int issued = 0;
    bool ok = true;
    for (int c = 0; c < nch; ++c) {
      const int st = c % kNST;
      if (c >= kNST) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->empty[st], ((c - kNST) / kNST) & 1));
        if (!ok) break;
      }
      if (lane == 0) {
        uint8_t* q = sm + st * kStage;
        uint64_t* bar = &bars->full[st];
        mbar_expect_tx(bar, kStage);
        const int z = t0 + c * kC;
        for (int sb = 0; sb < 2; ++sb) {
          tma_load_3d(q + sb * kSub, &tq, sb * 64, h, z, bar);
          tma_load_3d(q + kTile + sb * kSub, &tk, sb * 64, h, z, bar);
          tma_load_3d(q + 2 * kTile + sb * kSub, &tv, sb * 64, h, z, bar);
        }
      }
      issued = c + 1;
    }
    if (!ok && lane == 0) {                  // let the loads in flight land before exiting
      flag(status, HYB_DEVERR_TIMEOUT);
      for (int c = max(0, issued - kNST); c < issued; ++c)
        mbar_wait(&bars->full[c % kNST], (c / kNST) & 1, 100000000ull);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA warp
    // Issue order per chunk c: (d)_c, (b)_c, (a)_c, then (c)_{c-1} -- the output update of
    // the previous chunk goes last so the next state update never waits for P's conversion.
    bool ok = true;
    // descriptors built once; every MMA below adds an offset (see desc_add)
    const uint32_t sm0 = smem_u32(sm);
    const uint64_t mn0 = sw128_desc(sm0, kSub, 1024);          // MN-major, 64-row sub-tiles
    const uint64_t km0 = sw128_desc(sm0, 16, 1024);            // K-major
    const uint64_t st0 = sw128_desc(sm0 + kOffS, 16384, 1024); // S^T (bf16)
    auto issue_c = [&](int c) {                  // (c) O^T += V^T tril(P)^T of chunk c
      const int st = c % kNST, pb = c & 1;
      const uint32_t vo = st * kStage + 2 * kTile, po = kOffP + pb * kSub;
      if (lane == 0) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc_mma(tmem + kColO + pb * 64, desc_add(mn0, vo + k * 2048), desc_add(km0, po + k * 32),
                 kIdescC, 1);
        tc_commit(&bars->o_ready[pb]);
        tc_commit(&bars->empty[st]);
      }
      __syncwarp();
    };
    for (int c = 0; c < nch && ok; ++c) {
      const int st = c % kNST, ob = c & 1;
      uint8_t* qs = sm + st * kStage;
      uint8_t* ks = qs + kTile;
      uint8_t* vs = ks + kTile;
      const uint32_t qo = st * kStage, ko = qo + kTile, vo = ko + kTile;   // byte offsets in sm
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->full[st], (c / kNST) & 1));
      if (!ok) break;
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
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_read, c & 1));   // S of chunk c-1 read
      if (!ok) break;
      if (lane == 0) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)              // (d) S += K^T V
          tc_mma(tmem + kColS, desc_add(mn0, ko + k * 2048), desc_add(mn0, vo + k * 2048),
                 kIdescD, 1);
        tc_commit(&bars->s_ready);
      }
      if (c >= 2) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_free[ob], ((c - 2) >> 1) & 1));
        if (!ok) break;
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_written, c & 1));   // bf16 S^T ready
      if (!ok) break;
      if (lane == 0) {
        tc_fence_after();
        const uint32_t od = tmem + kColO + ob * 64;
#pragma unroll
        for (int k = 0; k < 8; ++k) {            // (b) O^T = S^T Q^T
          const uint32_t boff = (k >> 2) * kSub + (k & 3) * 32;
          tc_mma(od, desc_add(st0, k * 2048), desc_add(km0, qo + boff), kIdescB, k != 0);
        }
        tc_commit(&bars->b_done);
#pragma unroll
        for (int k = 0; k < 8; ++k) {            // (a) P = Q K^T
          const uint32_t off = (k >> 2) * kSub + (k & 3) * 32;
          tc_mma(tmem + kColP + ob * 64, desc_add(km0, qo + off), desc_add(km0, ko + off), kIdescA,
                 k > 0);
        }
        tc_commit(&bars->p_ready[ob]);
      }
      __syncwarp();
      if (c >= 1) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_written[(c - 1) & 1], ((c - 1) >> 1) & 1));
        if (!ok) break;
        issue_c(c - 1);
      }
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_written[(nch - 1) & 1], ((nch - 1) >> 1) & 1));
      if (ok) issue_c(nch - 1);
    }
    if (!ok && lane == 0) {                  // let every issued MMA finish before exiting
      flag(status, HYB_DEVERR_TIMEOUT);
      tc_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------ conversion warps
    // Warps 0-3 carry the state chain and P; warps 4-7 only write outputs, so a late output
    // never holds up the next state update. Warp w reaches TMEM lanes 32 * (w % 4) ...
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;                 // TMEM lane of this thread
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    bool ok = true;
    if (warp < 4) {
      const uint32_t soff0 = (row >> 3) * 1024;          // k-row group of the S^T operand
      // bf16 copy of 8 consecutive state values
      auto pack8 = [](const float* v) {
        return make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                          pack_bf16(v[6], v[7]));
      };
      // this thread's part of the S^T operand: k-row `row`, value columns 8 * ch ..; MN
      // block ch / 8
      auto put8 = [&](int ch, const uint4& w) {
        *reinterpret_cast<uint4*>(s_hi + (ch >> 3) * 16384 + soff0 + sw128_off(row & 7, ch & 7)) = w;
      };
      {                                                  // initial state, 32 columns at a time
#pragma unroll 1
        for (int part = 0; part < 4; ++part) {
          const int j0 = part * 32;
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 x = zero_start ? make_float4(0.f, 0.f, 0.f, 0.f)
                                        : *reinterpret_cast<const float4*>(Sg + (int64_t)row * kD + j0 + e);
            v[e] = x.x; v[e + 1] = x.y; v[e + 2] = x.z; v[e + 3] = x.w;
          }
          tmem_st32(tl + kColS + j0, v);
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) put8(part * 4 + ch, pack8(v + ch * 8));
        }
        tmem_st_wait();
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->s_read);
        mbar_arrive(&bars->s_written);
      }
      for (int c = 0; c < nch; ++c) {
        const bool last = c == nch - 1;
        // ---- new state: read it from TMEM; write the bf16 copy once (b) has used the old one
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_ready, c & 1));
        if (!ok) break;
        tc_fence_after();
        if (last) {
#pragma unroll 1
          for (int part = 0; part < 4; ++part) {
            const int j0 = part * 32;
            float v[32];
            tmem_ld32(tl + kColS + j0, v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(Sg + (int64_t)row * kD + j0 + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
          }
          tc_fence_before();
          mbar_arrive(&bars->s_read);
        } else {
          // hold the new state (as bf16) in registers and release TMEM: the next (d) may run
          uint4 w[16];
#pragma unroll
          for (int part = 0; part < 4; ++part) {
            float v[32];
            tmem_ld32(tl + kColS + part * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) w[part * 4 + ch] = pack8(v + ch * 8);
          }
          tc_fence_before();
          mbar_arrive(&bars->s_read);
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->b_done, c & 1));
          if (!ok) break;
#pragma unroll
          for (int ch = 0; ch < 16; ++ch) put8(ch, w[ch]);
          fence_async_smem();
        }
        tc_fence_before();
        mbar_arrive(&bars->s_written);
        // ---- tril(P) -> shared (K-major [t][t']), buffer c & 1
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_ready[c & 1], (c >> 1) & 1));
        if (!ok) break;
        tc_fence_after();
        {
          uint8_t* const pt = p_tile + (c & 1) * kSub;
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {
            float v[32];
            tmem_ld32(tl + kColP + (c & 1) * 64 + hf * 32, v);
            tmem_ld_wait();
            if (lane < 16) {
              const int t = quarter * 16 + lane;         // M = 64 layout: lanes 0..15 of each quarter
#pragma unroll
              for (int ch = 0; ch < 4; ++ch) {
                uint32_t wp[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int tp = hf * 32 + ch * 8 + 2 * e;
                  wp[e] = pack_bf16(tp <= t ? v[ch * 8 + 2 * e] : 0.f, tp + 1 <= t ? v[ch * 8 + 2 * e + 1] : 0.f);
                }
                *reinterpret_cast<uint4*>(pt + sw128_off(t, hf * 4 + ch)) = make_uint4(wp[0], wp[1], wp[2], wp[3]);
              }
            }
          }
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->p_written[c & 1]);
      }
    } else {
      // O^T of chunk cc -> global: this thread owns value dim j = row, all 64 tokens. Full
      // chunks go through staging buffer cc & 1 and a TMA store issued by one thread; before
      // a buffer is written again, that thread has seen the store that used it read it.
      const bool issuer = warp == 4 && lane == 0;
      for (int cc = 0; cc < nch && ok; ++cc) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_ready[cc & 1], (cc >> 1) & 1));
        if (!ok) break;
        tc_fence_after();
        float v[64];
        tmem_ld32(tl + kColO + (cc & 1) * 64, v);
        tmem_ld32(tl + kColO + (cc & 1) * 64 + 32, v + 32);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&bars->o_free[cc & 1]);              // TMEM buffer free for (b) of cc + 2
        const int nvalid = min(kC, n - cc * kC);
        if (nvalid < kC) {                               // partial chunk: direct stores
          __nv_bfloat16* o = out + ((int64_t)(t0 + cc * kC) * H + h) * kD + row;
          const int64_t step = (int64_t)H * kD;          // one token further
#pragma unroll
          for (int e = 0; e < 64; ++e) {
            if (e < nvalid) *o = __float2bfloat16_rn(v[e]);
            o += step;
          }
          continue;
        }
        const int sb = cc & 1;
        if (cc >= 2) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_stage_free[sb], ((cc - 2) >> 1) & 1));
          if (!ok) break;
        }
        // staging tile: two [64 tokens][64 j] SW128 sub-tiles (j halves), row = token; this
        // thread's j sits in 16-byte chunk (j & 63) / 8 at byte (j & 7) * 2
        uint8_t* const ob = o_stage + sb * kTile + (row >> 6) * kSub + (row & 7) * 2;
        const uint32_t jc = (row & 63) >> 3;
#pragma unroll
        for (int t = 0; t < 64; ++t)
          *reinterpret_cast<__nv_bfloat16*>(ob + sw128_off(t, jc)) = __float2bfloat16_rn(v[t]);
        fence_async_smem();
        mbar_arrive(&bars->o_staged[sb]);
        if (issuer) {
          if (!mbar_wait(&bars->o_staged[sb], (cc >> 1) & 1)) { ok = false; break; }
          tma_store_3d(&to, o_stage + sb * kTile, 0, h, t0 + cc * kC);
          tma_store_3d(&to, o_stage + sb * kTile + kSub, 64, h, t0 + cc * kC);
          bulk_commit();
          bulk_wait_read<1>();                           // the previous chunk's store has read
          if (cc >= 1) mbar_arrive(&bars->o_stage_free[sb ^ 1]);
        }
      }
      if (issuer) bulk_wait<0>();                        // every store complete before exit
    }
    if (!ok && lane == 0) flag(status, HYB_DEVERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
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
  if (B == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv, mo;
  const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)H, (uint64_t)(T > 0 ? T : 1)};
  const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)H * kD * 2};
  const uint32_t box[3] = {64, 1, (uint32_t)kC};
  if (!encode_tmap_bf16(&mq, q, 3, dims, strides, box) ||
      !encode_tmap_bf16(&mk, k, 3, dims, strides, box) ||
      !encode_tmap_bf16(&mv, v, 3, dims, strides, box) ||
      !encode_tmap_bf16(&mo, out, 3, dims, strides, box))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem((const void*)linear_prefill_tc_kernel, kSmem);
  if (e != cudaSuccess) return e;
  linear_prefill_tc_kernel<<<dim3(H, B), kThreads, kSmem, s>>>(
      mq, mk, mv, mo, static_cast<__nv_bfloat16*>(out), cu, ctx, pool, NS, slots, reset, H, status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace hyb
