// Causal prefill attention over the paged KV cache on the tensor cores (tcgen05 + TMEM +
// TMA), bf16, D = 128.
//
// Page: "推理框架适配Hybrid Model：KV Cache管理与算子调度实战", §2.3 -- prefill runs a
// FlashAttention-type kernel; the result it must equal is causal softmax attention, here
// read through the per-request block table (§2.1) so a cached prefix is attended as well.
//
// GB300 design. One CTA per (pair of 128-query tiles, head, request); heavy (late) pairs
// are scheduled first. Warp roles: two TMA warps (K ring, V ring), one MMA-issuing thread, a
// landing warp and two softmax warpgroups, one per query tile, one thread per query row (the
// row's max and sum stay in that thread). K and V come straight from the paged pool: each
// 128-key tile is eight 16-token blocks, each fetched with two TMA boxes (16 rows x 64
// columns, SW128) at the row the block table names (a block of bs tokens is bs / 16 such
// 16-row pieces); each TMA warp reads the block ids 32 pieces at a time and shares the rows
// with shuffles. Per key tile j and query tile t:
//   S_t = Q_t K_j^T   128 x 128 x 128  A = Q_t (K-major), B = K_j (K-major)  -> TMEM
//   O_t += P_t V_j    128 x 128 x 128  A = P_t (TMEM),    B = V_j (MN-major) -> TMEM
// TMEM holds S_0 | S_1 | O_0 | O_1 (4 x 128 columns). The softmax threads read S_t, write
// bf16 P_t into the first 64 columns of the same S_t region, and P V reads it from there:
// P never touches shared memory. The MMA thread issues, per key tile,
//   P_0 V_j, Q_0 K_{j+1}^T, P_1 V_j, Q_1 K_{j+1}^T
// so the tensor core works on one query tile while the other tile's softmax runs; the
// tensor pipe executes in issue order, so Q_t K_{j+1}^T overwrites P_t only after P_t V_j
// has read it, and its completion (the "S full" barrier) also tells the softmax threads
// that O_t is up to date. O stays in TMEM; a row is rescaled only when its running max
// grows by more than 2^8 (exponents stay <= 2^8, exact after the final division).
//
// tcgen05.mma returns only once the tensor pipe has taken the instruction (the issuing
// thread runs an MMA or two ahead of the pipe), so any wait or commit on that thread between
// two groups of MMAs idles the pipe for its whole latency (measured ~50-120 cycles each).
// The MMA thread therefore does nothing per key step but wait for P_t and commit S_t; the
// ring bookkeeping (data landed, slots free) runs on the landing warp (see Bars).
//
// Sliding window (window > 0, a query at position i sees keys i - window < p <= i): each
// query tile walks the key tiles from the one holding its first query's window start;
// blocks before the pair's window start are neither looked up nor loaded (their V rows are
// zeroed in shared memory instead), and the mask adds the lower bound. A row can see no
// key at all in its first tile; its exponent base is held at 0 until it sees one, so those
// P are 0.
#include <cuda_bf16.h>

#include "tc.cuh"

namespace hyb {
namespace {

constexpr int kBM = 128, kBN = 128, kD = 128;
constexpr int kSubQ = 128 * 128;             // [128 rows][64 cols] bf16 sub-tile = 16 KiB
constexpr int kTile = 2 * kSubQ;             // [128][128] bf16 = 32 KiB
constexpr int kNK = 2, kNV = 3;              // K and V ring depths (226 KiB in all)
constexpr int kOffQ = 0;                     // two query tiles
constexpr int kOffK = kOffQ + 2 * kTile;
constexpr int kOffV = kOffK + kNK * kTile;
constexpr int kOffBar = kOffV + kNV * kTile;
constexpr int kSmem = kOffBar + 1024 + 1024;  // barriers + 1 KiB alignment slack
constexpr int kNSW = 8;                      // softmax warps: 4 per query tile
constexpr int kWarpTmaK = kNSW, kWarpTmaV = kNSW + 1, kWarpMma = kNSW + 2, kWarpLand = kNSW + 3;
constexpr int kNSF = 4;                      // "step done" ring (see Bars)
constexpr int kThreads = (kNSW + 4) * 32;    // three full warpgroups
// Register split (setmaxnreg): the launch gives 384 threads x 168 registers (three warps
// per SM sub-partition). The producer warpgroup drops to 104 and the two softmax warpgroups
// rise to 200: 2 x 128 x 200 + 128 x 104 = 64 512 <= 64 512 registers of the launch, and
// (200 + 200 + 104) x 32 = 16 128 <= 16 384 per sub-partition.
constexpr uint32_t kRegsSoftmax = 200, kRegsProducer = 104;
constexpr uint32_t kTmemCols = 512;          // S_0/P_0 | S_1/P_1 | O_0 | O_1
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.f;
constexpr int kTailGroups = 16;              // (request, head) groups scheduled heavy first together

constexpr uint32_t kIdescQK = idesc_bf16(128, 128, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, 0, 1);   // A = P from TMEM

// The MMA-issuing thread does nothing per key step but wait for P_t (pfull) and commit S_t
// (sfull): tcgen05.mma blocks until the tensor pipe takes it, so every other wait or commit
// on that thread idles the pipe. The ring bookkeeping is done by other warps:
//  - the landing warp waits for V_j and K_{j+1} to land (and zeroes V rows a partially
//    valid last piece leaves stale) before it adds its arrival to pfull[t] for key tile j;
//  - a ring slot is free once the key step that read it is done. The step before key tile j
//    is done when its last MMA, Q_t K_j^T of the last query tile t reading key tile j,
//    completes (the commit on sfull[t] covers every earlier MMA); the landing warp waits for
//    that S (the softmax needs it before P_j anyway) and arrives on stepf[(j - jA) % kNSF].
//    Four slots: a producer waiting for a step can never see its slot two phases on.
struct Bars {
  uint64_t qfull, kfull[kNK], vfull[kNV], stepf[kNSF];
  uint64_t sfull[2], pfull[2], odone[2], drain;    // per query tile
};

// Paired fp32 arithmetic (one instruction for two lanes of a float2) and a three-input max:
// the softmax threads spend most of their issue slots on per-score work.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Whole warp: rows [r0, r1) of a [128 keys][128] bf16 V tile (two SW128 sub-tiles) := 0.
__device__ __forceinline__ void zero_v_rows(uint8_t* tile, int r0, int r1, int lane) {
  for (int e = lane; e < (r1 - r0) * 16; e += 32) {
    const int r = r0 + e / 16, sb = (e >> 3) & 1, ch = e & 7;
    *reinterpret_cast<uint4*>(tile + sb * kSubQ + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
  }
}

// Key-tile range [lo, hi) of one query tile and its key bound.
struct TileRange {
  int lo, hi, kv_end;
};

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, __nv_bfloat16* __restrict__ out,
                  const int32_t* __restrict__ bt, const int32_t* __restrict__ cu,
                  const int32_t* __restrict__ ctx, int H, int NB, int MB, int rsh,
                  float scale_log2, int window, unsigned* status) {
  // CTAs start in linear block order. Each (request, head) group's pairs run heavy first,
  // group after group, so a group's K/V tiles are re-read from L2. The last kTailGroups
  // groups (64 MiB of K/V at 8192 tokens) are interleaved heavy first across all of them,
  // so the final wave holds light pairs instead of a late group's heavy ones.
  const int np = gridDim.x, G = gridDim.y * gridDim.z;
  const int lin = blockIdx.x + np * (blockIdx.y + gridDim.y * blockIdx.z);
  const int gt = min(kTailGroups, G), head_ctas = (G - gt) * np;
  int pt, grp;
  if (lin < head_ctas) {
    grp = lin / np;
    pt = np - 1 - lin % np;
  } else {
    const int l = lin - head_ctas;
    grp = G - gt + l % gt;
    pt = np - 1 - l / gt;
  }
  const int h = grp % gridDim.y, b = grp / gridDim.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = cu[b], n = cu[b + 1] - t0;
  const int q0 = pt * 2 * kBM;                         // first query of the pair
  if (q0 >= n) return;
  const int c0 = ctx ? ctx[b] : 0;
  const bool two = q0 + kBM < n;                       // second query tile present
  TileRange tr[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qt = q0 + t * kBM;
    const int rows = max(0, min(kBM, n - qt));
    const int key_lo = window > 0 ? max(0, c0 + qt - window + 1) : 0;
    tr[t].kv_end = c0 + qt + rows;                     // keys the tile's last query sees
    tr[t].hi = (tr[t].kv_end + kBN - 1) / kBN;
    tr[t].lo = key_lo / kBN;
  }
  if (!two) tr[1].lo = tr[1].hi = tr[0].hi;            // empty range
  const int jA = tr[0].lo, jB = two ? tr[1].hi : tr[0].hi;   // union of the two ranges
  const int nloc = jB - jA;
  const int kv_end = two ? tr[1].kv_end : tr[0].kv_end;
  const int blk_lo = (window > 0 ? max(0, c0 + q0 - window + 1) : 0) / 16;
  const int32_t* btrow = bt + (int64_t)b * MB;
  if ((kv_end + 15) / 16 > (MB << rsh)) {             // in 16-token pieces
    if (tid == 0) flag(status, HYB_DEVERR_BAD_BLOCK);
    return;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(sm + kOffBar);
  __shared__ uint32_t tmem_base;

  if (warp == kWarpMma) {
    if (lane == 0) {
      mbar_init(&bars->qfull, 1);
      for (int i = 0; i < kNK; ++i) mbar_init(&bars->kfull[i], 1);
      for (int i = 0; i < kNV; ++i) mbar_init(&bars->vfull[i], 1);
      for (int i = 0; i < kNSF; ++i) mbar_init(&bars->stepf[i], 1);
      for (int t = 0; t < 2; ++t) {
        mbar_init(&bars->sfull[t], 1);
        mbar_init(&bars->pfull[t], 128 + 1);          // softmax threads + landing warp
        mbar_init(&bars->odone[t], 1);
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
  uint8_t* const q_s = sm + kOffQ;

  if (warp >= kNSW) {                               // producer warpgroup
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsProducer));
    if (warp == kWarpTmaK || warp == kWarpTmaV) {
      // ------------------------------------------------------------ TMA warps (K ring, V ring)
      // Two independent producers so K can run ahead of V (K is needed one step earlier).
      const bool isk = warp == kWarpTmaK;
      const CUtensorMap* map = isk ? &tk : &tv;
      const int depth = isk ? kNK : kNV;
      uint8_t* const ring = sm + (isk ? kOffK : kOffV);
      uint64_t* const fullb = isk ? bars->kfull : bars->vfull;
      bool ok = true;
      int issued = 0;
      if (lane == 0) {
        tma_prefetch_desc(map);
        if (isk) {                                       // both query tiles (rows past T read 0)
          tma_prefetch_desc(&tq);
          mbar_expect_tx(&bars->qfull, 2 * kTile);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            tma_load_3d(q_s + t * kTile, &tq, 0, h, t0 + q0 + t * kBM, &bars->qfull);
            tma_load_3d(q_s + t * kTile + kSubQ, &tq, 64, h, t0 + q0 + t * kBM, &bars->qfull);
          }
        }
      }
      int ids = -1;                                      // pool rows of 4 tiles' pieces, one per lane
      for (int jj = 0; jj < nloc; ++jj) {                // local tile index, key tile jA + jj
        if ((jj & 3) == 0) {
          const int lb = (jA + jj) * 8 + lane;             // 16-token piece of the sequence
          ids = -1;
          if (lb >= blk_lo && lb * 16 < kv_end) {
            const int pb = btrow[lb >> rsh];
            if (pb < 0 || pb >= NB) flag(status, HYB_DEVERR_BAD_BLOCK);
            else ids = ((pb * H + h) << (4 + rsh)) + ((lb & ((1 << rsh) - 1)) << 4);
          }
        }
        int blk[8];
        int nbox = 0;
#pragma unroll
        for (int bi = 0; bi < 8; ++bi) {
          blk[bi] = __shfl_sync(0xffffffffu, ids, (jj & 3) * 8 + bi);
          nbox += blk[bi] >= 0 ? 2 : 0;
        }
        const int slot = jj % depth;
        if (jj >= depth) {
          // the slot held K_{jj-kNK} (read by the Q K^T of the step before key tile jj-kNK)
          // or V_{jj-kNV} (read by the P V of its own step): free once that step is done
          const int m = isk ? jj - kNK : jj - kNV + 1;
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->stepf[m % kNSF], (m / kNSF) & 1));
          if (!ok) break;
        }
        // V rows that hold no key of this call must be finite (P is 0 there, but 0 x NaN is
        // NaN): the pieces that are not loaded are zeroed here, before the loads; the rows
        // past kv_end inside a partially valid last piece by the landing warp.
        const int kb = (jA + jj) * kBN;
        const int vhead = jj == 0 ? blk_lo * 16 - kb : 0;
        const int vtail16 = min(kBN, (kv_end - kb + 15) & ~15);
        if (!isk && (vhead > 0 || vtail16 < kBN)) {
          zero_v_rows(ring + slot * kTile, 0, vhead, lane);
          zero_v_rows(ring + slot * kTile, vtail16, kBN, lane);
          fence_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          uint8_t* dst = ring + slot * kTile;
          mbar_expect_tx(&fullb[slot], nbox * 2048);
#pragma unroll
          for (int bi = 0; bi < 8; ++bi)
            if (blk[bi] >= 0) {
              const int y = blk[bi];
              tma_load_2d(dst + bi * 2048, map, 0, y, &fullb[slot]);
              tma_load_2d(dst + kSubQ + bi * 2048, map, 64, y, &fullb[slot]);
            }
        }
        issued = jj + 1;
      }
      if (!ok && lane == 0) {                            // let the loads in flight land
        flag(status, HYB_DEVERR_TIMEOUT);
        for (int j = max(0, issued - depth); j < issued; ++j)
          mbar_wait(&fullb[j % depth], (j / depth) & 1, 100000000ull);
      }
    } else if (warp == kWarpLand) {
      // ------------------------------------------------------------ landing warp
      // Per key tile j: (1) the step before it is done -> stepf; (2) once V_j and K_{j+1} have
      // landed, one arrival on pfull[t] per query tile t that reads V_j (the MMA thread waits
      // for P_t anyway). It gates pfull, so it is never two phases behind on any barrier.
      // every phase of each barrier is observed in order (K_0 too), so a parity wait never
      // mistakes a phase two on for the one it waits for
      const int lo0 = tr[0].lo, hi0 = tr[0].hi, lo1 = tr[1].lo, hi1 = tr[1].hi;
      bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->kfull[0], 0));
      for (int jj = 0; jj < nloc && ok; ++jj) {
        const int j = jA + jj;
        // the last query tile reading key tile j (tile 1 unless its range misses j); its
        // S_j is number j - lo of that tile
        const bool b = j >= lo1 && j < hi1;
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->sfull[b ? 1 : 0], (j - (b ? lo1 : lo0)) & 1));
        if (!ok) break;
        if (lane == 0) mbar_arrive(&bars->stepf[jj % kNSF]);
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->vfull[jj % kNV], (jj / kNV) & 1));
        if (!ok) break;
        const int vtail = kv_end - j * kBN;
        if (vtail < kBN && (vtail & 15) != 0) {          // rows past kv_end in the last piece
          zero_v_rows(sm + kOffV + (jj % kNV) * kTile, vtail, min(kBN, (vtail + 15) & ~15), lane);
          fence_async_smem();
          __syncwarp();
        }
        if (jj + 1 < nloc) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->kfull[(jj + 1) % kNK], ((jj + 1) / kNK) & 1));
          if (!ok) break;
        }
        if (lane == 0) {
          if (j >= lo0 && j < hi0) mbar_arrive(&bars->pfull[0]);
          if (j >= lo1 && j < hi1) mbar_arrive(&bars->pfull[1]);
        }
        __syncwarp();
      }
      if (!ok && lane == 0) flag(status, HYB_DEVERR_TIMEOUT);
    } else if (warp == kWarpMma && lane == 0) {
      // ------------------------------------------------------------ MMA issue (one thread)
      // Per key tile j: wait for P_0 (which also means V_j and K_{j+1} have landed), P_0 V_j,
      // Q_0 K_{j+1}^T + commit; the same for tile 1. Nothing else: every extra instruction on
      // this thread between two MMA groups leaves the tensor pipe idle.
      bool ok = true;
      const uint64_t qdesc = sw128_desc(smem_u32(q_s), 16, 1024);
      const uint64_t kdesc = sw128_desc(smem_u32(sm + kOffK), 16, 1024);
      const uint64_t vdesc = sw128_desc(smem_u32(sm + kOffV), kSubQ, 1024);
      const int lo0 = tr[0].lo, hi0 = tr[0].hi, lo1 = tr[1].lo, hi1 = tr[1].hi;
      auto issue_qk = [&](int t, int ks) {               // S_t = Q_t K^T, K from ring slot ks
        tc_fence_after();
        const uint64_t qd = desc_add(qdesc, t * kTile);
        const uint64_t kd = desc_add(kdesc, ks * kTile);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * kSubQ + (k & 3) * 32;
          tc_mma(tmem + t * 128, desc_add(qd, off), desc_add(kd, off), kIdescQK, k > 0);
        }
        tc_commit(&bars->sfull[t]);
      };
      auto issue_pv = [&](int t, int vs, bool first) {   // O_t += P_t V_j
        tc_fence_after();
        const uint64_t vd = desc_add(vdesc, vs * kTile);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tc_mma_ta(tmem + kColO + t * 128, tmem + t * 128 + k * 8, desc_add(vd, k * 2048), kIdescPV,
                    (!first || k > 0) ? 1u : 0u);
      };
      ok = mbar_wait(&bars->qfull, 0) && mbar_wait(&bars->kfull[0], 0);
      if (ok) {
        if (lo0 <= jA && jA < hi0) issue_qk(0, 0);
        if (lo1 <= jA && jA < hi1) issue_qk(1, 0);
      }
      int npv0 = 0, npv1 = 0;                            // P V products issued per query tile
      for (int jj = 0; jj < nloc && ok; ++jj) {
        const int j = jA + jj, vs = jj % kNV, ks1 = (jj + 1) % kNK;
        const bool now0 = lo0 <= j && j < hi0, next0 = lo0 <= j + 1 && j + 1 < hi0;
        const bool now1 = lo1 <= j && j < hi1, next1 = lo1 <= j + 1 && j + 1 < hi1;
        if (now0) {
          ok = mbar_wait(&bars->pfull[0], npv0 & 1);
          if (!ok) break;
          issue_pv(0, vs, npv0 == 0);
          ++npv0;
        }
        if (next0) issue_qk(0, ks1);                     // tile 0 is active from jA on: now0
        else if (now0) tc_commit(&bars->odone[0]);       // O_0 complete
        if (now1) {
          ok = mbar_wait(&bars->pfull[1], npv1 & 1);
          if (!ok) break;
          issue_pv(1, vs, npv1 == 0);
          ++npv1;
        } else if (next1) {                              // tile 1's window starts at j + 1
          ok = mbar_wait(&bars->kfull[ks1], ((jj + 1) / kNK) & 1);
          if (!ok) break;
        }
        if (next1) issue_qk(1, ks1);
        else if (now1) tc_commit(&bars->odone[1]);       // O_1 complete
      }
      if (!ok) {
        flag(status, HYB_DEVERR_TIMEOUT);
        tc_commit(&bars->drain);
        mbar_wait(&bars->drain, 0, 100000000ull);
      }
    }
  } else {                                           // softmax warpgroups
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2, quarter = warp & 3;       // query tile, TMEM lane quarter
    const int r = quarter * 32 + lane;                 // query row of the tile = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_col = tl + t * 128, o_col = tl + kColO + t * 128;
    const int pos0 = c0 + q0 + t * kBM;                // position of the tile's first query
    const int qp = pos0 + r;                           // absolute query position
    const int qlo = window > 0 ? qp - window : -1;     // keys kp > qlo are in the window
    const TileRange my = t ? tr[1] : tr[0];            // (selects: no local-memory array)
    const int tkv_end = my.kv_end;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    int it = 0;
    for (int j = my.lo; j < my.hi && ok; ++j, ++it) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->sfull[t], it & 1));
      if (!ok) break;
      tc_fence_after();
      float x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_col + c * 32, x + c * 32);
      tmem_ld_wait();
      const int kbase = j * kBN;
      const bool masked = kbase + kBN - 1 > pos0 || kbase + kBN > tkv_end ||
                          (window > 0 && kbase <= pos0 + kBM - 1 - window);
      if (masked) {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int kp = kbase + c;
          x[c] = (kp <= qp && kp < tkv_end && kp > qlo) ? x[c] : -INFINITY;
        }
      }
      // row max of the raw scores (scale > 0 keeps the order): 8 independent chains of
      // three-input maxima
      float mp[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mp[i] = x[i];
#pragma unroll
      for (int c = 8; c + 16 <= 128; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) mp[i] = max3f(mp[i], x[c + i], x[c + 8 + i]);
#pragma unroll
      for (int i = 0; i < 8; ++i) mp[i] = fmaxf(mp[i], x[120 + i]);
      const float mx = max3f(max3f(mp[0], mp[1], mp[2]), max3f(mp[3], mp[4], mp[5]),
                             fmaxf(mp[6], mp[7])) * scale_log2;
      const float m_new = fmaxf(m_used, mx);
      const bool grow = m_new > m_used + kRescaleLog2 || (m_used == -INFINITY && m_new != -INFINITY);
      const float m_tgt = grow ? m_new : m_used;
      const float m_sub = m_tgt == -INFINITY ? 0.f : m_tgt;   // no key seen yet: P = 0
      // p = 2^(x * scale_log2 - m): one paired fma per two scores; sums in 4 paired chains
      uint32_t w[64];
      float2 sp[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sp[i] = make_float2(0.f, 0.f);
      const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(-m_sub, -m_sub);
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float2 y = fma2(make_float2(x[2 * c], x[2 * c + 1]), sc2, nm2);
        const float2 p = make_float2(fast_exp2(y.x), fast_exp2(y.y));
        sp[c & 3] = add2(sp[c & 3], p);
        w[c] = pack_bf16(p.x, p.y);
      }
      const float2 s01 = add2(add2(sp[0], sp[1]), add2(sp[2], sp[3]));
      const float ls = s01.x + s01.y;
      // O_t holds P V of every earlier tile: the S-full barrier that released this tile
      // completes after them (same tensor pipe, issued before)
      if (it >= 1 && __any_sync(0xffffffffu, grow)) {
        const float alpha = (grow && m_used != -INFINITY) ? fast_exp2(m_used - m_new) : 1.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {                  // warp-wide TMEM access, per-row factor
          float o[32];
          tmem_ld32(o_col + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32(o_col + c * 32, o);
        }
        if (grow) l *= alpha;
      }
      m_used = m_tgt;
      l += ls;
      tmem_st32u(s_col, w);                            // P_t: keys 0..127 as bf16 pairs
      tmem_st32u(s_col + 32, w + 32);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->pfull[t]);
    }
    if (ok && my.hi > my.lo)
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->odone[t], 0));
    if (ok && my.hi > my.lo) {
      // O_t / l -> bf16. Each warp stages its 32 rows in Q_t's shared memory (free once O_t
      // is complete: every MMA reading Q_t came before), 16-byte chunk c of row r at
      // r * 256 + (c ^ (r & 15)) * 16, then stores two whole rows (512 contiguous bytes) per
      // instruction instead of 32 rows 8 KiB apart.
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint8_t* const stage = q_s + t * kTile;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tmem_ld32(o_col + c * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 wv;
          wv.x = pack_bf16(o[e] * inv, o[e + 1] * inv);
          wv.y = pack_bf16(o[e + 2] * inv, o[e + 3] * inv);
          wv.z = pack_bf16(o[e + 4] * inv, o[e + 5] * inv);
          wv.w = pack_bf16(o[e + 6] * inv, o[e + 7] * inv);
          const int ch = (c * 32 + e) / 8;                 // 16-byte chunk 0..15 of the row
          *reinterpret_cast<uint4*>(stage + r * 256 + ((ch ^ (r & 15)) << 4)) = wv;
        }
      }
      __syncwarp();
      const int rows = n - (q0 + t * kBM);                 // rows of this tile in the prompt
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int rr = quarter * 32 + 2 * i + (lane >> 4), ch = lane & 15;
        if (rr < rows) {
          const uint4 wv = *reinterpret_cast<const uint4*>(stage + rr * 256 + ((ch ^ (rr & 15)) << 4));
          *reinterpret_cast<uint4*>(out + ((int64_t)(t0 + q0 + t * kBM + rr) * H + h) * kD + ch * 8) = wv;
        }
      }
    } else if (!ok && lane == 0) {
      flag(status, HYB_DEVERR_TIMEOUT);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool prefill_tc_supported(int dtype, int D) { return dtype == HYB_BF16 && D == kD; }

cudaError_t launch_prefill_tc(void* out, const void* q, const void* kc, const void* vc,
                              const int32_t* bt, const int32_t* cu, const int32_t* ctx, int B,
                              int T, int max_q_len, int H, int NB, int MB, int bs, float scale,
                              int window, unsigned* status, cudaStream_t s) {
  if (B == 0 || max_q_len == 0 || T <= 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  const uint64_t qdims[3] = {(uint64_t)kD, (uint64_t)H, (uint64_t)T};
  const uint64_t qstr[2] = {(uint64_t)kD * 2, (uint64_t)H * kD * 2};
  const uint32_t qbox[3] = {64, 1, (uint32_t)kBM};
  const uint64_t cdims[2] = {(uint64_t)kD, (uint64_t)NB * H * bs};
  const uint64_t cstr[1] = {(uint64_t)kD * 2};
  const uint32_t cbox[2] = {64, 16};
  if (!encode_tmap_bf16(&mq, q, 3, qdims, qstr, qbox) ||
      !encode_tmap_bf16(&mk, kc, 2, cdims, cstr, cbox) ||
      !encode_tmap_bf16(&mv, vc, 2, cdims, cstr, cbox))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem((const void*)prefill_tc_kernel, kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((max_q_len + 2 * kBM - 1) / (2 * kBM), H, B);
  prefill_tc_kernel<<<grid, kThreads, kSmem, s>>>(mq, mk, mv, static_cast<__nv_bfloat16*>(out), bt,
                                                  cu, ctx, H, NB, MB, log2_int(bs / 16),
                                                  scale * 1.4426950408889634f, window, status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace hyb
