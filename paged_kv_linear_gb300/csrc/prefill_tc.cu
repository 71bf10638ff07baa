// Causal prefill attention over the paged KV cache on the tensor cores (tcgen05 + TMEM +
// TMA), bf16, D = 128.
//
// Page: "推理框架适配Hybrid Model：KV Cache管理与算子调度实战", §2.3 -- prefill runs a
// FlashAttention-type kernel; the result it must equal is causal softmax attention, here
// read through the per-request block table (§2.1) so a cached prefix is attended as well.
//
// GB300 design. One CTA per (128-query tile, head, request); heavy (late) query tiles are
// scheduled first. Warp roles: two TMA warps (K ring, V ring), an MMA warp and eight
// softmax warps. K and V come straight from the paged pool: each 128-key tile is eight
// 16-token blocks, each fetched with two TMA boxes (16 rows x 64 columns, SW128) at the row
// the block table names, into a 3-deep K ring and a 2-deep V ring; each TMA warp reads the
// block ids 32 at a time (four tiles) and shares them with shuffles. Per key tile:
//   S = Q K^T     128 x 128 x 128  A = Q (K-major), B = K (K-major)    -> TMEM, 2 buffers
//   O += P V      128 x 128 x 128  A = P (TMEM),    B = V (MN-major)   -> TMEM
// Each query row is split over two softmax threads (two warps, 64 columns each) that swap
// their partial row max through shared memory once per tile. They apply the causal/length
// mask, keep the running max and sum, and write bf16 P back into TMEM (two buffers), where
// P V reads it as its A operand: P never touches shared memory, which leaves the tensor
// core's shared-memory bandwidth to Q, K and V. O stays in TMEM; a row is rescaled only
// when its running max grows by more than 2^8 (exponents stay <= 2^8, exact after the
// final division by the row sum). S is double-buffered so Q K^T of tile j+2 and P V of
// tile j run on the tensor core while the softmax threads exponentiate tile j+1; they wait
// for P V only to reuse a P buffer (two tiles back) or to rescale O.
//
// Sliding window (window > 0, a query at position i sees keys i - window < p <= i): the
// key tiles start at the one holding the window start of the tile's first query, blocks
// before that start are neither looked up nor loaded (their V rows are zeroed in shared
// memory instead), and the mask adds the lower bound. A row can then see no key at all in
// its first tiles; its exponent base is held at 0 until it sees one, so those P are 0.
#include <cuda_bf16.h>

#include "tc.cuh"

namespace hyb {
namespace {

constexpr int kBM = 128, kBN = 128, kD = 128;
constexpr int kSubQ = 128 * 128;             // [128 rows][64 cols] bf16 sub-tile = 16 KiB
constexpr int kTile = 2 * kSubQ;             // [128][128] bf16 = 32 KiB
constexpr int kNK = 3, kNV = 2;              // K and V ring depths
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTile;
constexpr int kOffV = kOffK + kNK * kTile;
constexpr int kOffBar = kOffV + kNV * kTile;
constexpr int kSmem = kOffBar + 4096 + 1024;
constexpr int kNSW = 8;                      // softmax warps: 2 per TMEM lane quarter
constexpr int kWarpTmaK = kNSW, kWarpTmaV = kNSW + 1, kWarpMma = kNSW + 2;
constexpr int kThreads = (kNSW + 3) * 32;
constexpr uint32_t kTmemCols = 512;          // S0 | S1 | O | P0 | P1 (P: bf16 pairs)
constexpr uint32_t kColO = 256, kColP = 384;
constexpr float kRescaleLog2 = 8.f;

constexpr uint32_t kIdescQK = idesc_bf16(128, 128, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, 0, 1);   // A = P from TMEM

struct Bars {
  uint64_t qfull, kfull[kNK], kempty[kNK], vfull[kNV], vempty[kNV];
  uint64_t sfull[2], pfull[2], odone[2], drain;   // handshakes per tile parity
  uint64_t pair[4][2];                       // the two warps of a lane quarter, per parity
  float red[2][2][kBM];                      // row-half partial max per parity; final sums
};

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, __nv_bfloat16* __restrict__ out,
                  const int32_t* __restrict__ bt, const int32_t* __restrict__ cu,
                  const int32_t* __restrict__ ctx, int H, int NB, int MB, float scale_log2,
                  int window, unsigned* status) {
  const int qt = gridDim.x - 1 - blockIdx.x;           // heavy tiles first
  const int h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = cu[b], n = cu[b + 1] - t0;
  const int q0 = qt * kBM;
  if (q0 >= n) return;
  const int c0 = ctx ? ctx[b] : 0;
  const int rows = min(kBM, n - q0);
  const int kv_end = c0 + q0 + rows;                   // keys the tile's last query sees
  const int nkv = (kv_end + kBN - 1) / kBN;
  const int pos0 = c0 + q0;                            // position of the tile's first query
  const int key_lo = window > 0 ? max(0, pos0 - window + 1) : 0;   // first key any row sees
  const int jlo = key_lo / kBN;                        // first key tile
  const int nloc = nkv - jlo;                          // key tiles this CTA walks
  const int blk_lo = key_lo / 16;                      // first block looked up and loaded
  const int32_t* btrow = bt + (int64_t)b * MB;
  if ((kv_end + 15) / 16 > MB) {
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
      for (int i = 0; i < kNK; ++i) { mbar_init(&bars->kfull[i], 1); mbar_init(&bars->kempty[i], 1); }
      for (int i = 0; i < kNV; ++i) { mbar_init(&bars->vfull[i], 1); mbar_init(&bars->vempty[i], 1); }
      mbar_init(&bars->sfull[0], 1);
      mbar_init(&bars->sfull[1], 1);
      mbar_init(&bars->pfull[0], kNSW * 32);
      mbar_init(&bars->pfull[1], kNSW * 32);
      mbar_init(&bars->odone[0], 1);
      mbar_init(&bars->odone[1], 1);
      mbar_init(&bars->drain, 1);
      for (int qq = 0; qq < 4; ++qq) {
        mbar_init(&bars->pair[qq][0], 64);
        mbar_init(&bars->pair[qq][1], 64);
      }
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

  if (warp == kWarpTmaK || warp == kWarpTmaV) {
    // ------------------------------------------------------------ TMA warps (K ring, V ring)
    // Two independent producers so K can run ahead of V (K is needed one tile earlier).
    const bool isk = warp == kWarpTmaK;
    const CUtensorMap* map = isk ? &tk : &tv;
    const int depth = isk ? kNK : kNV;
    uint8_t* const ring = sm + (isk ? kOffK : kOffV);
    uint64_t* const fullb = isk ? bars->kfull : bars->vfull;
    uint64_t* const emptyb = isk ? bars->kempty : bars->vempty;
    bool ok = true;
    int issued = 0;
    if (lane == 0) {
      tma_prefetch_desc(map);
      if (isk) {
        tma_prefetch_desc(&tq);
        mbar_expect_tx(&bars->qfull, kTile);
        tma_load_3d(q_s, &tq, 0, h, t0 + q0, &bars->qfull);
        tma_load_3d(q_s + kSubQ, &tq, 64, h, t0 + q0, &bars->qfull);
      }
    }
    int ids = -1;                                      // block ids of 4 tiles, one per lane
    for (int jj = 0; jj < nloc; ++jj) {                // jj: local tile index, j = jlo + jj
      if ((jj & 3) == 0) {
        const int lb = (jlo + jj) * 8 + lane;
        ids = -1;
        if (lb >= blk_lo && lb * 16 < kv_end) {
          ids = btrow[lb];
          if (ids < 0 || ids >= NB) {
            flag(status, HYB_DEVERR_BAD_BLOCK);
            ids = -1;
          }
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
        ok = __all_sync(0xffffffffu, mbar_wait(&emptyb[slot], ((jj - depth) / depth) & 1));
        if (!ok) break;
      }
      if (lane == 0) {
        uint8_t* dst = ring + slot * kTile;
        mbar_expect_tx(&fullb[slot], nbox * 2048);
#pragma unroll
        for (int bi = 0; bi < 8; ++bi)
          if (blk[bi] >= 0) {
            const int y = (blk[bi] * H + h) * 16;
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
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA warp
    bool ok = true;
    // descriptors built once; every MMA below adds a compile-time offset
    const uint64_t qdesc = sw128_desc(smem_u32(q_s), 16, 1024);
    const uint64_t kdesc = sw128_desc(smem_u32(sm + kOffK), 16, 1024);
    const uint64_t vdesc = sw128_desc(smem_u32(sm + kOffV), kSubQ, 1024);
    auto issue_qk = [&](int j) -> bool {           // S[j%2] = Q K_j^T (j: local tile index)
      const int ks = j % kNK;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->kfull[ks], (j / kNK) & 1))) return false;
      if (lane == 0) {
        tc_fence_after();
        const uint64_t kd = desc_add(kdesc, ks * kTile);
        const uint32_t sd = tmem + (j & 1) * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * kSubQ + (k & 3) * 32;
          tc_mma(sd, desc_add(qdesc, off), desc_add(kd, off), kIdescQK, k > 0);
        }
        tc_commit(&bars->sfull[j & 1]);
        tc_commit(&bars->kempty[ks]);
      }
      __syncwarp();
      return true;
    };
    ok = __all_sync(0xffffffffu, mbar_wait(&bars->qfull, 0));
    if (ok) ok = issue_qk(0);
    if (ok && nloc > 1) ok = issue_qk(1);
    for (int j = 0; j < nloc && ok; ++j) {           // local tile index; keys from (jlo+j)*128
      const int vs = j % kNV;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->pfull[j & 1], (j >> 1) & 1));
      if (!ok) break;
      // softmax of tile j is done with S buffer j&1: queue Q K_{j+2} first so the softmax
      // threads have their next-but-one scores early (an MMA issue blocks while the tensor
      // core is busy, so issue order is execution order)
      if (j + 2 < nloc) {
        ok = issue_qk(j + 2);
        if (!ok) break;
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->vfull[vs], (j / kNV) & 1));
      if (!ok) break;
      uint8_t* v_s = sm + kOffV + vs * kTile;
      // V rows that were not loaded := 0 (P is 0 there, but stale shared memory may hold
      // NaN): rows past kv_end in the last tile, rows before the window's first block
      const int kb = (jlo + j) * kBN;
      const int head = j == 0 ? blk_lo * 16 - kb : 0;
      const int tail = kv_end - kb;
      if (head > 0 || tail < kBN) {
        auto zero_rows = [&](int r0, int r1) {
          for (int e = lane; e < (r1 - r0) * 16; e += 32) {
            const int r = r0 + e / 16, sb = (e >> 3) & 1, ch = e & 7;
            *reinterpret_cast<uint4*>(v_s + sb * kSubQ + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
          }
        };
        if (head > 0) zero_rows(0, head);
        if (tail < kBN) zero_rows(tail, kBN);
        fence_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        tc_fence_after();
        const uint64_t vd = desc_add(vdesc, vs * kTile);
        const uint32_t pt = tmem + kColP + (j & 1) * 64;
#pragma unroll
        for (int k = 0; k < 8; ++k)                // O += P V_j, P read from TMEM buffer j&1
          tc_mma_ta(tmem + kColO, pt + k * 8, desc_add(vd, k * 2048), kIdescPV,
                    (j > 0 || k > 0) ? 1u : 0u);
        tc_commit(&bars->odone[j & 1]);
        tc_commit(&bars->vempty[vs]);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) {
      flag(status, HYB_DEVERR_TIMEOUT);
      tc_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int quarter = warp & 3, hf = warp >> 2;      // TMEM lane quarter, column half
    const int r = quarter * 32 + lane;                 // query row of the tile = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const int qp = pos0 + r;                           // absolute query position
    const int qlo = window > 0 ? qp - window : -1;     // keys kp > qlo are in the window
    const int c0h = hf * 64;                           // this thread's 64 columns
    float m_used = -INFINITY, l = 0.f;                 // l: this half's share of the row sum
    bool ok = true;
    // swap a value with the other half of this row (exchange number idx); bounded wait
    auto pair_swap = [&](int idx, float v, float& other) -> bool {
      bars->red[idx & 1][hf][r] = v;
      mbar_arrive(&bars->pair[quarter][idx & 1]);
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->pair[quarter][idx & 1], (idx >> 1) & 1)))
        return false;
      other = bars->red[idx & 1][hf ^ 1][r];
      return true;
    };
    for (int j = 0; j < nloc && ok; ++j) {            // local tile index; keys from (jlo+j)*128
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->sfull[j & 1], (j >> 1) & 1));
      if (!ok) break;
      tc_fence_after();
      float x[64];
      tmem_ld32(tl + (j & 1) * 128 + c0h, x);
      tmem_ld32(tl + (j & 1) * 128 + c0h + 32, x + 32);
      tmem_ld_wait();
      const int kbase = (jlo + j) * kBN + c0h;
      const bool masked = kbase + 63 > pos0 || kbase + 64 > kv_end ||
                          (window > 0 && kbase <= pos0 + kBM - 1 - window);
      if (masked) {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int kp = kbase + c;
          x[c] = (kp <= qp && kp < kv_end && kp > qlo) ? x[c] : -INFINITY;
        }
      }
      // partial max of the raw scores (scale > 0 keeps the order): 8 independent chains
      float mp[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mp[i] = x[i];
#pragma unroll
      for (int c = 8; c < 64; ++c) mp[c & 7] = fmaxf(mp[c & 7], x[c]);
      float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                       fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      float mx_other;
      ok = pair_swap(j, mx, mx_other);
      if (!ok) break;
      mx = fmaxf(mx, mx_other) * scale_log2;
      const float m_new = fmaxf(m_used, mx);
      const bool grow = m_new > m_used + kRescaleLog2 || (m_used == -INFINITY && m_new != -INFINITY);
      const float m_tgt = grow ? m_new : m_used;
      const float m_sub = m_tgt == -INFINITY ? 0.f : m_tgt;   // no key seen yet: P = 0
      // exponentials of this tile first: they do not depend on P V of the previous tile.
      // p = 2^(x * scale_log2 - m) as one fma per element; sum in 8 independent chains.
      uint32_t w[32];
      float sp[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) sp[i] = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = fast_exp2(fmaf(x[2 * c], scale_log2, -m_sub));
        const float p1 = fast_exp2(fmaf(x[2 * c + 1], scale_log2, -m_sub));
        sp[c & 7] += p0 + p1;
        w[c] = pack_bf16(p0, p1);
      }
      const float ls = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
      if (j >= 2) {                                    // P V_{j-2} done: P buffer j&1 free
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->odone[j & 1], ((j - 2) >> 1) & 1));
        if (!ok) break;
      }
      if (j >= 1 && __any_sync(0xffffffffu, grow)) {   // rescale O once P V_{j-1} is in
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->odone[(j - 1) & 1], ((j - 1) >> 1) & 1));
        if (!ok) break;
        tc_fence_after();
        const float alpha = (grow && m_used != -INFINITY) ? fast_exp2(m_used - m_new) : 1.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {                  // warp-wide TMEM access, per-row factor
          float o[32];
          tmem_ld32(tl + kColO + c0h + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32(tl + kColO + c0h + c * 32, o);
        }
        if (grow) l *= alpha;
      }
      m_used = m_tgt;
      l += ls;
      tc_fence_after();
      tmem_st32u(tl + kColP + (j & 1) * 64 + hf * 32, w);   // keys c0h..c0h+63 as bf16 pairs
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->pfull[j & 1]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->odone[(nloc - 1) & 1], ((nloc - 1) >> 1) & 1));
    float l_other = 0.f;
    if (ok) ok = pair_swap(nloc, l, l_other);          // row sum = both halves' shares
    if (ok) {
      const float lt = l + l_other;
      tc_fence_after();
      const bool store = q0 + r < n;
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      __nv_bfloat16* orow = out + ((int64_t)(t0 + q0 + r) * H + h) * kD + c0h;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float o[32];
        tmem_ld32(tl + kColO + c0h + c * 32, o);
        tmem_ld_wait();
        if (store) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 wv;
            wv.x = pack_bf16(o[e] * inv, o[e + 1] * inv);
            wv.y = pack_bf16(o[e + 2] * inv, o[e + 3] * inv);
            wv.z = pack_bf16(o[e + 4] * inv, o[e + 5] * inv);
            wv.w = pack_bf16(o[e + 6] * inv, o[e + 7] * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + e) = wv;
          }
        }
      }
    } else if (lane == 0) {
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
                              int T, int max_q_len, int H, int NB, int MB, float scale,
                              int window, unsigned* status, cudaStream_t s) {
  if (B == 0 || max_q_len == 0 || T <= 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  const uint64_t qdims[3] = {(uint64_t)kD, (uint64_t)H, (uint64_t)T};
  const uint64_t qstr[2] = {(uint64_t)kD * 2, (uint64_t)H * kD * 2};
  const uint32_t qbox[3] = {64, 1, (uint32_t)kBM};
  const uint64_t cdims[2] = {(uint64_t)kD, (uint64_t)NB * H * 16};
  const uint64_t cstr[1] = {(uint64_t)kD * 2};
  const uint32_t cbox[2] = {64, 16};
  if (!encode_tmap_bf16(&mq, q, 3, qdims, qstr, qbox) ||
      !encode_tmap_bf16(&mk, kc, 2, cdims, cstr, cbox) ||
      !encode_tmap_bf16(&mv, vc, 2, cdims, cstr, cbox))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem((const void*)prefill_tc_kernel, kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((max_q_len + kBM - 1) / kBM, H, B);
  prefill_tc_kernel<<<grid, kThreads, kSmem, s>>>(mq, mk, mv, static_cast<__nv_bfloat16*>(out), bt,
                                                  cu, ctx, H, NB, MB, scale * 1.4426950408889634f,
                                                  window, status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace hyb
