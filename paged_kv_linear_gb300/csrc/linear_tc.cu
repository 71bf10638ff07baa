// Chunked linear-attention prefill on the tensor cores (tcgen05 + TMEM + TMA), bf16 q/k/v,
// D = 128, chunk C = 64, fp32 state.
//
// Page: "推理框架适配Hybrid Model：KV Cache管理与算子调度实战", §2.1 (state update
// S <- S + k (outer) v, output q.S), §2.3 (state zeroed at request start, accumulated in
// prefill, kept in fp32) and §2.4 (chunks carry the state; chunk boundaries aligned).
// Per chunk c of a (request, head), with S the fp32 state at the chunk start:
//     O_c = Q_c S + tril(Q_c K_c^T) V_c        S <- S + K_c^T V_c
//
// GB300 design. Each (request, head) chain is sequential, and there are often not many more
// chains than SMs (8 x 32 = 256 chains on 152 SMs would leave a second wave two-thirds
// full). So one CTA per SM, all resident at once (cooperative launch), takes an equal share
// of all chunks laid end to end; a chain cut between two CTAs hands its state over through
// the state pool (see "work split" below). Within a CTA the runs follow one another without
// draining the pipeline. Warp roles: one TMA warp streams Q/K/V chunks through a 3-stage ring (SW128
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
  uint64_t published;        // state warps' pool writes of a run that hands its state over
};

// ------------------------------------------------------------------ work split
// Units are the (request, head) chains, in order u = b * H + h; unit u has nch(b) chunks.
// Laid end to end they occupy G chunk positions. CTA p takes positions [p*L, (p+1)*L) with
// L = max(longest chain, ceil(G / P)) (McNaughton's wrap-around rule for preemptive
// scheduling on P machines), so no chain crosses more than one CTA boundary. A chain cut
// at the boundary (p+1)*L is run in two parts, its first chunks by CTA p+1 FIRST and the
// rest by CTA p LAST: the first part is no longer than the work CTA p does before its last
// part, so the state it hands over (through the state pool) is ready when it is needed.
// A handoff is announced by a flag that names the call: the call's epoch (a counter that a
// one-thread kernel bumps right before every launch, in stream order, so graph replays get
// fresh epochs too) and the launch's grid id (distinct for launches that run at the same
// time). A waiting CTA accepts only its own call's value, never one left by another call.
constexpr int kMaxCtas = 256;                // grid limit (one CTA per SM)
constexpr int kRegions = 64;                 // flag sets, chosen by the launch's grid id
// handoff flags: entry p holds the tag of the call whose CTA p has written the state of the
// chain it cut (at its first boundary) to the pool.
__device__ unsigned long long g_lin_handoff[kRegions][kMaxCtas];
__device__ unsigned g_lin_epoch;

__global__ void linear_handoff_epoch_kernel() {
  pdl_wait();                                // everything before it in the stream is done
  g_lin_epoch += 1;
}

struct Plan {
  int head_u, head_end;      // chain run first, chunks [0, head_end); -1: none
  int full_u0, full_u1;      // chains run whole, in order
  int tail_u, tail_begin;    // chain run last, chunks [tail_begin, nch); -1: none
};

__device__ __forceinline__ int chunks_of(const int32_t* cu, int b) {
  const int n = cu[b + 1] - cu[b];
  return n > 0 ? (n + kC - 1) / kC : 0;
}

__device__ __forceinline__ int warp_incl_scan(int x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Run by one whole warp; every lane returns the same plan for CTA p of P.
__device__ Plan make_plan(const int32_t* cu, int B, int H, int P, int p, int lane) {
  long long total = 0;
  int longest = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int nc = b0 + lane < B ? chunks_of(cu, b0 + lane) : 0;
    total += __reduce_add_sync(0xffffffffu, (unsigned)nc);
    longest = max(longest, (int)__reduce_max_sync(0xffffffffu, (unsigned)nc));
  }
  const long long G = total * H;
  const long long L = max((long long)longest, (G + P - 1) / P);
  const long long s = (long long)p * L, e = min(s + L, G);
  Plan pl{-1, 0, 0, 0, -1, 0};
  if (s >= G) return pl;
  // locate positions s and e: request b holds [base + H*excl, base + H*incl)
  int us = -1, offs = 0, ue = -1, offe = 0;
  long long base = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    const int nc = b < B ? chunks_of(cu, b) : 0;
    const int incl = warp_incl_scan(nc, lane);
    const long long lo = base + (long long)H * (incl - nc), hi = base + (long long)H * incl;
    const bool in_s = nc > 0 && s >= lo && s < hi, in_e = nc > 0 && e >= lo && e < hi;
    const unsigned ms = __ballot_sync(0xffffffffu, in_s), me = __ballot_sync(0xffffffffu, in_e);
    const int u_s = in_s ? b * H + (int)((s - lo) / nc) : 0, o_s = in_s ? (int)((s - lo) % nc) : 0;
    const int u_e = in_e ? b * H + (int)((e - lo) / nc) : 0, o_e = in_e ? (int)((e - lo) % nc) : 0;
    if (ms) {
      const int l = __ffs(ms) - 1;
      us = __shfl_sync(0xffffffffu, u_s, l);
      offs = __shfl_sync(0xffffffffu, o_s, l);
    }
    if (me) {
      const int l = __ffs(me) - 1;
      ue = __shfl_sync(0xffffffffu, u_e, l);
      offe = __shfl_sync(0xffffffffu, o_e, l);
    }
    base += (long long)H * __shfl_sync(0xffffffffu, incl, 31);
  }
  if (offs > 0) {
    pl.head_u = us;
    pl.head_end = chunks_of(cu, us / H) - offs;
    pl.full_u0 = us + 1;
  } else {
    pl.full_u0 = us;
  }
  if (e >= G) {
    pl.full_u1 = B * H;
  } else if (offe > 0) {
    pl.tail_u = ue;
    pl.tail_begin = chunks_of(cu, ue / H) - offe;
    pl.full_u1 = ue;
  } else {
    pl.full_u1 = ue;
  }
  return pl;
}

// A contiguous run of one chain's chunks, [c0, c1).
struct Seg {
  int h, t0, n, c0, c1;
  float* S;                  // the chain's state in the pool
  bool zero_start;           // c0 == 0 and the request is reset
  bool wait_handoff;         // c0 > 0: the state comes from the CTA that ran chunks [0, c0)
  bool publish;              // c1 < nch: hand the state over at the end
};

// Makes run [c0, c1) (c1 < 0: to the end) of chain `unit`; false if the chain has no rows
// or its request is invalid (reported once, in the prologue).
__device__ __forceinline__ bool make_run(int unit, int c0, int c1, const int32_t* cu,
                                         const int32_t* ctx, const int32_t* slots,
                                         const uint8_t* reset, float* pool, int NS, int H,
                                         Seg& s) {
  const int b = unit / H;
  const int nc = chunks_of(cu, b);
  const int slot = slots[b];
  if (nc == 0 || slot < 0 || slot >= NS || (ctx && ctx[b] % kC != 0)) return false;
  s.h = unit - b * H;
  s.t0 = cu[b];
  s.n = cu[b + 1] - s.t0;
  s.c0 = c0;
  s.c1 = c1 < 0 ? nc : c1;
  s.S = pool + ((int64_t)slot * H + s.h) * kD * kD;
  s.zero_start = c0 == 0 && reset && reset[b];
  s.wait_handoff = c0 > 0;
  s.publish = s.c1 < nc;
  return true;
}

// Position in this CTA's runs: the first chain's part, the whole chains, the last chain's
// part, in that order. Every warp walks its own copy.
struct Walk {
  int stage = 0, u = -1;
};
__device__ __forceinline__ bool next_run(Walk& w, const Plan& pl, const int32_t* cu,
                                         const int32_t* ctx, const int32_t* slots,
                                         const uint8_t* reset, float* pool, int NS, int H,
                                         Seg& s) {
  while (true) {
    if (w.stage == 0) {
      w.stage = 1;
      w.u = pl.full_u0;
      if (pl.head_u >= 0 && make_run(pl.head_u, 0, pl.head_end, cu, ctx, slots, reset, pool, NS, H, s))
        return true;
    } else if (w.stage == 1) {
      if (w.u < pl.full_u1) {
        if (make_run(w.u++, 0, -1, cu, ctx, slots, reset, pool, NS, H, s)) return true;
      } else {
        w.stage = 2;
      }
    } else if (w.stage == 2) {
      w.stage = 3;
      if (pl.tail_u >= 0 && make_run(pl.tail_u, pl.tail_begin, -1, cu, ctx, slots, reset, pool, NS, H, s))
        return true;
    } else {
      return false;
    }
  }
}

__device__ __forceinline__ unsigned long long grid_id() {
  unsigned long long g;
  asm volatile("mov.u64 %0, %%gridid;" : "=l"(g));
  return g;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint4 pack8(const float* v) {     // bf16 copy of 8 values
  return make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                    pack_bf16(v[6], v[7]));
}

// This thread's 16-byte piece ch (value columns 8 ch ..) of the S^T operand: k-row `row`,
// MN block ch / 8, SW128 layout.
__device__ __forceinline__ void put8(uint8_t* s_t, int row, int ch, const uint4& w) {
  *reinterpret_cast<uint4*>(s_t + (ch >> 3) * 16384 + (row >> 3) * 1024 + sw128_off(row & 7, ch & 7)) = w;
}

// Starting state of run `sg`, row `row` (one state warp thread) -> TMEM lane `tl`, and its
// bf16 copy -> the S^T operand s_t (which (b) must no longer be reading). A run that
// continues a chain first waits until the CTA that ran the chain's start has published it
// with this call's tag `want` (on expiry: reported, and the pool's contents are used as
// they are).
__device__ __forceinline__ void load_start(const Seg& sg, uint8_t* s_t, uint32_t tl, int row,
                                           const unsigned long long* handoff_flag,
                                           unsigned long long want, unsigned* status) {
  if (sg.wait_handoff) {
    const uint64_t t0 = global_ns();
    while (ld_acquire_u64(handoff_flag) != want) {
      if (global_ns() - t0 > 2000000000ull) {
        flag(status, HYB_DEVERR_TIMEOUT);
        break;
      }
      __nanosleep(100);
    }
  }
#pragma unroll
  for (int part = 0; part < 4; ++part) {
    const int j0 = part * 32;
    float v[32];
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const float4 x = sg.zero_start ? make_float4(0.f, 0.f, 0.f, 0.f)
                                     : __ldcg(reinterpret_cast<const float4*>(sg.S + (int64_t)row * kD + j0 + e));
      v[e] = x.x; v[e + 1] = x.y; v[e + 2] = x.z; v[e + 3] = x.w;
    }
    tmem_st32(tl + kColS + j0, v);
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) put8(s_t, row, part * 4 + ch, pack8(v + ch * 8));
  }
  tmem_st_wait();
  fence_async_smem();
}

__global__ void __launch_bounds__(kThreads, 1)
linear_prefill_tc_kernel(const __grid_constant__ CUtensorMap tq,
                         const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv,
                         const __grid_constant__ CUtensorMap to, __nv_bfloat16* __restrict__ out,
                         const int32_t* __restrict__ cu, const int32_t* __restrict__ ctx,
                         float* __restrict__ pool, int NS, const int32_t* __restrict__ slots,
                         const uint8_t* __restrict__ reset, int B, int H, unsigned* status) {
  const int p = blockIdx.x, P = gridDim.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ Plan plan_sh;
  __shared__ uint32_t tmem_base;

  // prologue: invalid requests are reported; a reset request without rows gets a zero state
  for (int b = p; b < B; b += P) {
    const int slot = slots[b];
    if (slot < 0 || slot >= NS) {
      if (tid == 0) flag(status, HYB_DEVERR_BAD_STATE);
      continue;
    }
    if (ctx && ctx[b] % kC != 0) {
      if (tid == 0) flag(status, HYB_DEVERR_MISALIGNED);
      continue;
    }
    if (cu[b + 1] - cu[b] <= 0 && reset && reset[b]) {
      float4* S = reinterpret_cast<float4*>(pool + (int64_t)slot * H * kD * kD);
      for (int e = tid; e < H * kD * kD / 4; e += kThreads) S[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (warp == 0) {
    const Plan pl = make_plan(cu, B, H, P, p, lane);
    if (lane == 0) plan_sh = pl;
  }
  __syncthreads();
  if (plan_sh.head_u < 0 && plan_sh.tail_u < 0 && plan_sh.full_u0 >= plan_sh.full_u1) return;
  const unsigned long long gid = grid_id();
  unsigned long long* const handoff = g_lin_handoff[gid % kRegions];
  const unsigned long long tag =
      ((unsigned long long)*reinterpret_cast<volatile unsigned*>(&g_lin_epoch) << 32) | (gid & 0xffffffffull);
  Walk walk;
#define NEXT_RUN(sg) next_run(walk, plan_sh, cu, ctx, slots, reset, pool, NS, H, sg)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(sm + kOffBar);

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
      mbar_init(&bars->published, 128);
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
    int c = 0;
    bool ok = true;
    Seg sg;
    while (ok && NEXT_RUN(sg)) {
      for (int ci = sg.c0; ci < sg.c1; ++ci, ++c) {
        const int st = c % kNST;
        if (c >= kNST) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->empty[st], ((c - kNST) / kNST) & 1));
          if (!ok) break;
        }
        if (lane == 0) {
          uint8_t* q = sm + st * kStage;
          uint64_t* bar = &bars->full[st];
          mbar_expect_tx(bar, kStage);
          const int z = sg.t0 + ci * kC;
          for (int sb = 0; sb < 2; ++sb) {
            tma_load_3d(q + sb * kSub, &tq, sb * 64, sg.h, z, bar);
            tma_load_3d(q + kTile + sb * kSub, &tk, sb * 64, sg.h, z, bar);
            tma_load_3d(q + 2 * kTile + sb * kSub, &tv, sb * 64, sg.h, z, bar);
          }
        }
      }
    }
    if (!ok && lane == 0) {                  // let the loads in flight land before exiting
      flag(status, HYB_DEVERR_TIMEOUT);
      for (int i = max(0, c - kNST); i < c; ++i)
        mbar_wait(&bars->full[i % kNST], (i / kNST) & 1, 100000000ull);
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
    int c = 0;
    Seg sg;
    while (ok && NEXT_RUN(sg)) {
      for (int ci = sg.c0; ci < sg.c1; ++ci, ++c) {
        const int st = c % kNST, ob = c & 1;
        uint8_t* qs = sm + st * kStage;
        uint8_t* ks = qs + kTile;
        uint8_t* vs = ks + kTile;
        const uint32_t qo = st * kStage, ko = qo + kTile, vo = ko + kTile;   // byte offsets in sm
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->full[st], (c / kNST) & 1));
        if (!ok) break;
        const int nvalid = min(kC, sg.n - ci * kC);
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
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_read, c & 1));   // state of chunk c-1 read
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
    }
    if (ok && c > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_written[(c - 1) & 1], ((c - 1) >> 1) & 1));
      if (ok) issue_c(c - 1);
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
      Seg sg;
      bool have = NEXT_RUN(sg);
      if (have) {
        load_start(sg, s_hi, tl, row, &handoff[p + 1], tag, status);
        tc_fence_before();
        mbar_arrive(&bars->s_read);
        mbar_arrive(&bars->s_written);
      }
      int ci = sg.c0;
      for (int c = 0; have; ++c) {
        // ---- new state: read it from TMEM; write the bf16 copy once (b) has used the old one
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_ready, c & 1));
        if (!ok) break;
        tc_fence_after();
        if (ci == sg.c1 - 1) {
          // end of a run: the state goes to the pool (and is handed over if the chain goes
          // on in another CTA); the next run's starting state takes its place once (b) has
          // read the last copy
#pragma unroll 1
          for (int part = 0; part < 4; ++part) {
            const int j0 = part * 32;
            float v[32];
            tmem_ld32(tl + kColS + j0, v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(sg.S + (int64_t)row * kD + j0 + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
          }
          if (sg.publish) {                              // at most once per CTA (its first run)
            __threadfence();
            mbar_arrive(&bars->published);
            if (tid == 0) {
              if (mbar_wait(&bars->published, 0)) st_release_u64(&handoff[p], tag);
              else flag(status, HYB_DEVERR_TIMEOUT);
            }
          }
          have = NEXT_RUN(sg);
          ci = sg.c0;
          if (have) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars->b_done, c & 1));
            if (!ok) break;
            load_start(sg, s_hi, tl, row, &handoff[p + 1], tag, status);
          }
          tc_fence_before();
          mbar_arrive(&bars->s_read);
        } else {
          // hold the new state (as bf16) in registers and release TMEM: the next (d) may run;
          // write the copy once (b) has used the old one
          uint4 w[16];
#pragma unroll
          for (int part = 0; part < 4; ++part) {
            float v[32];
            tmem_ld32(tl + kColS + part * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) w[part * 4 + ch] = pack8(v + ch * 8);
          }
          ++ci;
          tc_fence_before();
          mbar_arrive(&bars->s_read);
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->b_done, c & 1));
          if (!ok) break;
#pragma unroll
          for (int ch = 0; ch < 16; ++ch) put8(s_hi, row, ch, w[ch]);
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
      // O^T of chunk c -> global: this thread owns value dim j = row, all 64 tokens. Full
      // chunks go through staging buffer f & 1 (f counts full chunks) and a TMA store issued
      // by one thread; before a buffer is written again, that thread has seen the store that
      // used it read it.
      const bool issuer = warp == 4 && lane == 0;
      int c = 0, f = 0;
      Seg sg;
      while (ok && NEXT_RUN(sg)) {
        for (int ci = sg.c0; ci < sg.c1; ++ci, ++c) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_ready[c & 1], (c >> 1) & 1));
          if (!ok) break;
          tc_fence_after();
          float v[64];
          tmem_ld32(tl + kColO + (c & 1) * 64, v);
          tmem_ld32(tl + kColO + (c & 1) * 64 + 32, v + 32);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&bars->o_free[c & 1]);               // TMEM buffer free for (b) of c + 2
          const int z = sg.t0 + ci * kC;
          const int nvalid = min(kC, sg.n - ci * kC);
          if (nvalid < kC) {                               // partial chunk: direct stores
            __nv_bfloat16* o = out + ((int64_t)z * H + sg.h) * kD + row;
            const int64_t step = (int64_t)H * kD;          // one token further
#pragma unroll
            for (int e = 0; e < 64; ++e) {
              if (e < nvalid) *o = __float2bfloat16_rn(v[e]);
              o += step;
            }
            continue;
          }
          const int sb = f & 1;
          if (f >= 2) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_stage_free[sb], ((f - 2) >> 1) & 1));
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
            if (!mbar_wait(&bars->o_staged[sb], (f >> 1) & 1)) { ok = false; break; }
            tma_store_3d(&to, o_stage + sb * kTile, 0, sg.h, z);
            tma_store_3d(&to, o_stage + sb * kTile + kSub, 64, sg.h, z);
            bulk_commit();
            bulk_wait_read<1>();                           // the previous chunk's store has read
            if (f >= 1) mbar_arrive(&bars->o_stage_free[sb ^ 1]);
          }
          ++f;
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
#undef NEXT_RUN
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
  e = launch_pdl(linear_handoff_epoch_kernel, dim3(1), dim3(1), 0, s);
  count_launch();
  if (e != cudaSuccess) return e;
  // One CTA per SM at most (the shared memory allows no more), all resident at once: a CTA
  // may wait for the state another CTA hands over, so the launch is cooperative.
  const int64_t units = (int64_t)B * H;
  const int grid = (int)std::min<int64_t>(std::min(num_sms(), kMaxCtas), units);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, linear_prefill_tc_kernel, mq, mk, mv, mo,
                         static_cast<__nv_bfloat16*>(out), cu, ctx, pool, NS, slots, reset, B, H,
                         status);
  count_launch();
  return e;
}

}  // namespace hyb
