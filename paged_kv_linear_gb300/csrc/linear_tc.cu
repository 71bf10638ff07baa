// Chunked linear-attention prefill on the tensor cores (tcgen05 + TMEM + TMA), bf16 q/k/v,
// D = 128, fp32 state.
//
// Page: "推理框架适配Hybrid Model：KV Cache管理与算子调度实战", §2.1 (state update
// S <- S + k (outer) v, output q.S), §2.3 (state zeroed at request start, accumulated in
// prefill, kept in fp32) and §2.4 (chunks carry the state; chunk boundaries aligned).
// Per chunk c of a (request, head), with S the fp32 state at the chunk start:
//     O_c = Q_c S + tril(Q_c K_c^T) V_c        S <- S + K_c^T V_c
// The result does not depend on where the chunks are cut, so the kernel cuts each call's
// rows into chunks of 128 (the call's start must still sit on a 64-token boundary, the
// chunk size of the interface): every product is then a 128 x 128 tile, the shape the
// tensor core runs best (a smaller N costs almost as many cycles per instruction).
//
// GB300 design. Each (request, head) chain is sequential, and there are often not many more
// chains than SMs (8 x 32 = 256 chains on 152 SMs would leave a second wave two-thirds
// full). So one CTA per SM, all resident at once (cooperative launch), takes an equal share
// of all chunks laid end to end; a chain cut between two CTAs hands its state over through
// the state pool (see "work split" below). Within a CTA the runs follow one another without
// draining the pipeline. Warp roles: one TMA warp streams Q/K/V chunks through a 2-stage
// ring (SW128 tiles, one "full" mbarrier per stage, one "empty" mbarrier per tile of a
// stage); one MMA warp issues the tensor-core work;
// four state warps carry the state and P; four output warps write O. The state lives in
// TMEM for the whole call and is accumulated in place. Per chunk (M x N x K, all 128):
//   (d) S  += K_c^T V_c      A = K^T (MN-major), B = V (MN-major)
//   (b) O   = Q_c S          A = Q (K-major), B = the state at the chunk start rounded to
//                            bf16 (MN-major, shared memory; the fp32 state stays in TMEM)
//   (a) P   = Q_c K_c^T      A = Q, B = K (both K-major), fp32 into TMEM
//   (c) O  += tril(P) V_c    A = tril(P) as bf16 in TMEM (written over P by the state
//                            warps), B = V (MN-major)
// Issue order per chunk: (a)_c, (d)_c, (b)_c, (c)_c. The state warps convert P_c while
// (d)_c and (b)_c run. Each tile of the chunk's ring stage is released after its own last
// MMA (K after (d), Q after (b), V after (c)) and reloaded in that order, so the loads of
// chunk c+2 start while chunk c is still computing. The tensor core runs the MMAs in order,
// so (a)_{c+1} overwrites P only after (c)_c has read it. The state chain is (d) -> read S
// from TMEM -> next (d): the state warps release the state as soon as it is in their
// registers ("S read") and write its bf16 copy for (b) once (b) has consumed the previous
// one ("S written"). O is double-buffered in TMEM; every handshake barrier has one phase in
// flight at most. Output rows go straight from registers to global memory (one thread per
// token row of 256 bytes).
#include <cuda_bf16.h>

#include "tc.cuh"

namespace hyb {
namespace {

constexpr int kC = 128, kD = 128;            // chunk rows, head dim
constexpr int kAlign = 64;                   // chunk size of the interface: call starts align to it
constexpr int kNST = 2;                      // Q/K/V ring stages
constexpr int kBoxRows = 16;                 // rows per TMA box; both column halves of a row
                                             // group are requested back to back
constexpr int kSub = 128 * 128;              // bytes of one [128 rows][64 cols] SW128 sub-tile
constexpr int kTile = 2 * kSub;              // [128][128] bf16 tile
constexpr int kStage = 3 * kTile;            // Q, K, V
constexpr int kOffS = kNST * kStage;         // state as bf16 ([128 i][128 j], MN-major B)
constexpr int kSTile = 128 * 128 * 2;
constexpr int kOffBar = kOffS + kSTile;
constexpr int kSmem = kOffBar + 256 + 1024;  // + slack for 1024-byte alignment
constexpr int kWarpTma = 8, kWarpMma = 9;
constexpr int kThreads = 10 * 32;
constexpr uint32_t kTmemCols = 512;          // S [0,128) | O x2 [128,384) | P [384,512)
constexpr uint32_t kColS = 0, kColO = 128, kColP = 384;

constexpr uint32_t kIdescD = idesc_bf16(128, 128, 1, 1);   // K^T, V: both MN-major
constexpr uint32_t kIdescB = idesc_bf16(128, 128, 0, 1);   // Q K-major, S MN-major
constexpr uint32_t kIdescA = idesc_bf16(128, 128, 0, 0);   // Q, K: K-major
constexpr uint32_t kIdescC = idesc_bf16(128, 128, 0, 1);   // tril(P) from TMEM, V MN-major

struct Bars {
  uint64_t full[kNST];
  uint64_t empty[3][kNST];          // per tile of a stage (Q, K, V): each frees after its last MMA
  uint64_t s_ready, s_read, b_done, s_written, drain;
  uint64_t p_ready, p_written;
  uint64_t o_ready[2], o_free[2];   // one per buffer parity
  uint64_t published;               // state warps' pool writes of a run that hands its state over
};
static_assert(sizeof(Bars) <= 256, "barriers overflow their shared-memory slot");

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
// time). A waiting CTA accepts only its own call's value, never one left by an earlier call.
// Epoch and flags live in the caller's workspace: hs[0] is the epoch, hs[1 + p] holds the tag
// of the call whose CTA p has written the state of the chain it cut (at its first boundary)
// to the pool. The library itself holds no handoff state, so calls with distinct workspaces
// never see each other's flags.
constexpr int kMaxCtas = kLinMaxCtas;        // grid limit (one CTA per SM)

__global__ void linear_handoff_epoch_kernel(unsigned long long* hs) {
  pdl_wait();                                // everything before it in the stream is done
  hs[0] += 1;
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
  if (nc == 0 || slot < 0 || slot >= NS || (ctx && ctx[b] % kAlign != 0)) return false;
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

// This thread's 16-byte piece ch (value columns 8 ch ..) of the bf16 state operand: row
// i = `row`, MN block ch / 8, SW128 layout ([j / 64][i / 8][i % 8][j % 64]).
__device__ __forceinline__ void put8(uint8_t* s_t, int row, int ch, const uint4& w) {
  *reinterpret_cast<uint4*>(s_t + (ch >> 3) * 16384 + (row >> 3) * 1024 + sw128_off(row & 7, ch & 7)) = w;
}

// Starting state of run `sg`, row `row` (one state warp thread) -> TMEM lane `tl`, and its
// bf16 copy -> the operand s_t (which (b) must no longer be reading). A run that continues
// a chain first waits until the CTA that ran the chain's start has published it with this
// call's tag `want` (on expiry: reported, and the pool's contents are used as they are).
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
                         const __grid_constant__ CUtensorMap tv, __nv_bfloat16* __restrict__ out,
                         const int32_t* __restrict__ cu, const int32_t* __restrict__ ctx,
                         float* __restrict__ pool, int NS, const int32_t* __restrict__ slots,
                         const uint8_t* __restrict__ reset, int B, int H,
                         unsigned long long* __restrict__ hs, unsigned* status) {
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
    if (ctx && ctx[b] % kAlign != 0) {
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
  unsigned long long* const handoff = hs + 1;
  const unsigned long long tag =
      (*reinterpret_cast<volatile unsigned long long*>(hs) << 32) | (gid & 0xffffffffull);
  Walk walk;
#define NEXT_RUN(sg) next_run(walk, plan_sh, cu, ctx, slots, reset, pool, NS, H, sg)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(sm + kOffBar);

  if (warp == kWarpMma) {
    if (lane == 0) {
      for (int s = 0; s < kNST; ++s) {
        mbar_init(&bars->full[s], 3);                // one arrival per tile, with its bytes
        for (int t = 0; t < 3; ++t) mbar_init(&bars->empty[t][s], 1);
      }
      mbar_init(&bars->s_ready, 1);
      mbar_init(&bars->b_done, 1);
      mbar_init(&bars->s_read, 128);               // state warps (0-3)
      mbar_init(&bars->s_written, 128);
      mbar_init(&bars->p_ready, 1);
      mbar_init(&bars->p_written, 128);            // state warps
      for (int i = 0; i < 2; ++i) {
        mbar_init(&bars->o_ready[i], 1);
        mbar_init(&bars->o_free[i], 128);          // output warps (4-7)
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
        uint8_t* q = sm + st * kStage;
        uint64_t* bar = &bars->full[st];
        const int z = sg.t0 + ci * kC;
        // Tiles in the order the MMAs release them: K after (d), Q after (b), V after (c).
        int t = 0;
#pragma unroll
        for (; t < 3; ++t) {
          const int tt = t == 0 ? 1 : (t == 1 ? 0 : 2);
          if (c >= kNST) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars->empty[tt][st], ((c - kNST) / kNST) & 1));
            if (!ok) break;
          }
          if (lane == 0) {
            const CUtensorMap* m = tt == 0 ? &tq : (tt == 1 ? &tk : &tv);
            mbar_expect_tx(bar, kTile);
            for (int r0 = 0; r0 < kC; r0 += kBoxRows)
              for (int sb = 0; sb < 2; ++sb)
                tma_load_3d(q + tt * kTile + sb * kSub + r0 * 128, m, sb * 64, sg.h, z + r0, bar);
          }
        }
        if (!ok) {                           // the tiles not issued arrive without bytes, so
          if (t > 0) {                       // the chunk's phase completes when its loads land
            if (lane == 0)
              for (int r = t; r < 3; ++r) mbar_arrive(bar);
            ++c;
          }
          break;
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
    bool ok = true;
    // descriptors built once; every MMA below adds an offset (see desc_add)
    const uint32_t sm0 = smem_u32(sm);
    const uint64_t mn0 = sw128_desc(sm0, kSub, 1024);          // MN-major: two 64-wide blocks
    const uint64_t km0 = sw128_desc(sm0, 16, 1024);            // K-major
    const uint64_t st0 = sw128_desc(sm0 + kOffS, 16384, 1024); // bf16 state (MN-major)
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
        if (lane == 0) {
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k) {            // (a) P = Q K^T (after (c) of c-1 read P)
            const uint32_t off = (k >> 2) * kSub + (k & 3) * 32;
            tc_mma(tmem + kColP, desc_add(km0, qo + off), desc_add(km0, ko + off), kIdescA, k > 0);
          }
          tc_commit(&bars->p_ready);
        }
        __syncwarp();
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_read, c & 1));   // state of chunk c-1 read
        if (!ok) break;
        if (lane == 0) {
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)              // (d) S += K^T V
            tc_mma(tmem + kColS, desc_add(mn0, ko + k * 2048), desc_add(mn0, vo + k * 2048), kIdescD, 1);
          tc_commit(&bars->s_ready);
          tc_commit(&bars->empty[1][st]);        // K's last use
        }
        if (c >= 2) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_free[ob], ((c - 2) >> 1) & 1));
          if (!ok) break;
        }
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_written, c & 1));   // bf16 state ready
        if (!ok) break;
        if (lane == 0) {
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k) {            // (b) O = Q S
            const uint32_t aoff = (k >> 2) * kSub + (k & 3) * 32;
            tc_mma(tmem + kColO + ob * 128, desc_add(km0, qo + aoff), desc_add(st0, k * 2048), kIdescB, k != 0);
          }
          tc_commit(&bars->b_done);
          tc_commit(&bars->empty[0][st]);        // Q's last use
        }
        __syncwarp();
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_written, c & 1));
        if (!ok) break;
        if (lane == 0) {
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)              // (c) O += tril(P) V
            tc_mma_ta(tmem + kColO + ob * 128, tmem + kColP + k * 8, desc_add(mn0, vo + k * 2048), kIdescC, 1);
          tc_commit(&bars->o_ready[ob]);
          tc_commit(&bars->empty[2][st]);        // V's last use
        }
        __syncwarp();
      }
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
        // ---- tril(P) as bf16 pairs over the first 64 columns of P (row t = this lane); (c)
        // waits for it right after (b), so P goes first
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_ready, c & 1));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {           // keys 64 half .. 64 half + 63
          uint32_t w[32];
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            float v[32];
            tmem_ld32(tl + kColP + half * 64 + q2 * 32, v);
            tmem_ld_wait();
            const int tp0 = half * 64 + q2 * 32;
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[q2 * 16 + e] = pack_bf16(tp0 + 2 * e <= row ? v[2 * e] : 0.f,
                                         tp0 + 2 * e + 1 <= row ? v[2 * e + 1] : 0.f);
          }
          tmem_st32u(tl + kColP + half * 32, w);         // reads of these columns are done
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_written);
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
      }
    } else {
      // O of chunk c -> global: this thread owns token row t = row, all 128 value columns
      int c = 0;
      Seg sg;
      while (ok && NEXT_RUN(sg)) {
        for (int ci = sg.c0; ci < sg.c1; ++ci, ++c) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_ready[c & 1], (c >> 1) & 1));
          if (!ok) break;
          tc_fence_after();
          uint32_t w[64];
#pragma unroll
          for (int part = 0; part < 4; ++part) {
            float v[32];
            tmem_ld32(tl + kColO + (c & 1) * 128 + part * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) w[part * 16 + e] = pack_bf16(v[2 * e], v[2 * e + 1]);
          }
          tc_fence_before();
          mbar_arrive(&bars->o_free[c & 1]);             // TMEM buffer free for (b) of c + 2
          if (row < min(kC, sg.n - ci * kC)) {
            uint4* o = reinterpret_cast<uint4*>(out + ((int64_t)(sg.t0 + ci * kC + row) * H + sg.h) * kD);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
          }
        }
      }
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
  return dtype == HYB_BF16 && D == kD && C == kAlign;
}

cudaError_t launch_linear_prefill_tc(void* out, const void* q, const void* k, const void* v,
                                     const int32_t* cu, const int32_t* ctx, float* pool, int NS,
                                     const int32_t* slots, const uint8_t* reset, int B, int T,
                                     int max_len, int H, int C, void* ws, unsigned* status,
                                     cudaStream_t s) {
  (void)max_len;
  (void)C;
  if (B == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)H, (uint64_t)(T > 0 ? T : 1)};
  const uint64_t strides[2] = {(uint64_t)kD * 2, (uint64_t)H * kD * 2};
  const uint32_t box[3] = {64, 1, (uint32_t)kBoxRows};
  if (!encode_tmap_bf16(&mq, q, 3, dims, strides, box) ||
      !encode_tmap_bf16(&mk, k, 3, dims, strides, box) ||
      !encode_tmap_bf16(&mv, v, 3, dims, strides, box))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem((const void*)linear_prefill_tc_kernel, kSmem);
  if (e != cudaSuccess) return e;
  unsigned long long* hs = static_cast<unsigned long long*>(ws);
  e = launch_pdl(linear_handoff_epoch_kernel, dim3(1), dim3(1), 0, s, hs);
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
  e = cudaLaunchKernelEx(&cfg, linear_prefill_tc_kernel, mq, mk, mv,
                         static_cast<__nv_bfloat16*>(out), cu, ctx, pool, NS, slots, reset, B, H,
                         hs, status);
  count_launch();
  return e;
}

}  // namespace hyb
