// Paged decode attention: split-K online softmax over 16-token KV blocks.
//
// Page: "推理框架适配Hybrid Model：KV Cache管理与算子调度实战", §2.3 (decode uses a
// PagedAttention-type kernel reading K/V through the block table) and §2.1 (a decode
// step of a Full layer costs O(S x D) and the KV cache is the bandwidth hog).
//
// Design (GB300): the work is pure HBM streaming -- every (block, head) K and V tile is
// a contiguous 16 x D run of the [NB][H][16][D] pool (4 KiB each at D=128, bf16), read
// once. A CTA owns one (row, head, split of 32 blocks) and 4 warps; each warp walks every
// 4th block of the split through its own 2-stage ring in shared memory, filled by the TMA
// engine (cp.async.bulk, one 4 KiB copy per tile, completion on an mbarrier). The small
// ring (64 KiB per CTA) fits three CTAs per SM, which on GB300 streams faster than deeper
// rings with fewer resident CTAs (measured over warps x stages x split sizes). Scores and the
// online softmax run in fp32 on the CUDA cores with warp shuffles; partial states
// (m, l, acc[D]) of the 4 warps merge in shared memory, and splits merge in a second
// small kernel (log-sum-exp combine). The split size is a constant number of blocks, so
// a request's result does not depend on the rest of the batch.
//
// The grid is (split, row, head) with the split index fastest. In a batch of mixed lengths
// most CTAs of the grid have no split to run; with the split index slowest, the long rows'
// later splits were dispatched behind planes of such empty CTAs and ran alone at the end.
//
// In a decode dispatch, a Full layer after the first reads its row length and block ids and
// requests its first K/V tiles before waiting for the previous kernel (which writes neither
// this layer's cache nor the batch metadata); q and the new row are read after the wait.
//
// The same kernel serves as the CUDA-core causal prefill for shapes without a
// tensor-core kernel (PREFILL = true: one row per packed query token, n = position + 1,
// one CTA walks all of the row's blocks).
//
// Sliding window (window > 0): a row sees keys [n - window, n). The splits cover only the
// blocks from the one holding n - window; earlier blocks and their block-table entries are
// never read, so an allocator may have released them.
#include <cuda_bf16.h>

#include "hyb_internal.cuh"

namespace hyb {

namespace {

#ifndef HYB_DECODE_NW
#define HYB_DECODE_NW 4
#endif
#ifndef HYB_DECODE_NST
#define HYB_DECODE_NST 2
#endif
#ifndef HYB_DECODE_BPS
#define HYB_DECODE_BPS 32
#endif
constexpr int kNW = HYB_DECODE_NW;    // warps per CTA
constexpr int kNST = HYB_DECODE_NST;  // ring stages per warp
constexpr int kBPS = HYB_DECODE_BPS;  // KV blocks per split (constant: batch-invariant results)

template <typename T>
struct Elt;
template <>
struct Elt<__nv_bfloat16> {
  static constexpr int VEC = 8;
  __device__ static void unpack(const uint4& u, float* f) {
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
  }
  __device__ static void store(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
};
template <>
struct Elt<float> {
  static constexpr int VEC = 4;
  __device__ static void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  __device__ static void store(float* p, float x) { *p = x; }
};

// Length handled for a row after host/device bound checks (identical in both kernels);
// MBt = block-table capacity in 16-token sub-tiles.
__device__ __forceinline__ int clamp_len(int n, int max_len, int MBt) {
  n = n < 0 ? 0 : n;
  n = n > max_len ? max_len : n;
  const int cap = MBt * kBlockSize;
  return n > cap ? cap : n;
}

// First key a row of n keys attends to.
__device__ __forceinline__ int window_lo(int n, int window) {
  return (window > 0 && n > window) ? n - window : 0;
}

// Splits of a decode row: ranges of kBPS blocks from the window's first block.
__device__ __forceinline__ int decode_splits(int n, int window) {
  const int nblk = (n + kBlockSize - 1) / kBlockSize;
  const int blk_lo = window_lo(n, window) / kBlockSize;
  return max(1, (nblk - blk_lo + kBPS - 1) / kBPS);
}

template <typename T, int D>
struct DecodeShape {
  static constexpr int VEC = Elt<T>::VEC;
  static constexpr int LPR = D / VEC;          // lanes covering one token row
  static constexpr int TPI = 32 / LPR;         // token rows per warp load
  static constexpr int ITER = kBlockSize / TPI;
  static constexpr int TILE = kBlockSize * D * (int)sizeof(T);
  static constexpr int SMEM = kNW * kNST * 2 * TILE + kNW * kNST * 8 + kNW * (D + 2) * 4;
  static_assert(LPR >= 2 && LPR <= 32 && ITER >= 1, "unsupported head_dim");
};

// WINDOW = false compiles the lower key bound away (window must then be 0).
template <typename T, int D, bool PREFILL, bool WINDOW>
__global__ void __launch_bounds__(kNW * 32)
paged_decode_kernel(T* __restrict__ out, const T* __restrict__ q, T* __restrict__ kc,
                    T* __restrict__ vc, const int32_t* __restrict__ bt,
                    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu,
                    const int32_t* __restrict__ ctx, int max_q, int H, int NB, int MB,
                    int rsh, int max_len, float scale_log2, int window, int max_splits,
                    float* __restrict__ ws_acc, float2* __restrict__ ws_ml,
                    const T* __restrict__ k_new, const T* __restrict__ v_new,
                    const int64_t* __restrict__ slot_map, int early, unsigned* status) {
  using E = Elt<T>;
  using S = DecodeShape<T, D>;
  constexpr int VEC = S::VEC, LPR = S::LPR, TPI = S::TPI, ITER = S::ITER, TILE = S::TILE;

  // early (decode after another layer of the same dispatch): no kernel before it in the
  // dispatch writes anything this layer reads (its cache, q, the new row, block table,
  // lengths), so it runs its whole K/V stream while the previous kernel drains and waits for
  // that kernel only before its first write of the shared split workspace or the output.
  if (!early) pdl_wait();                  // inputs may come from the previous kernel
  // decode: grid (splits, rows, H), the split index fastest; prefill: (rows, H, 1)
  const int h = PREFILL ? blockIdx.y : blockIdx.z, split = PREFILL ? 0 : blockIdx.x;
  int b, r, n_raw;                         // request, packed row of q/out, keys to attend
  if (PREFILL) {                           // grid.x = B * max_q: (request, query index)
    b = blockIdx.x / max_q;
    const int j = blockIdx.x - b * max_q;
    if (j >= cu[b + 1] - cu[b]) return;
    r = cu[b] + j;
    n_raw = (ctx ? ctx[b] : 0) + j + 1;
  } else {
    b = r = blockIdx.y;
    n_raw = seq_lens[r];
  }
  const int n = clamp_len(n_raw, max_len, MB << rsh);
  if (n != (n_raw < 0 ? 0 : n_raw) && split == 0 && threadIdx.x == 0)
    flag(status, n_raw > max_len ? HYB_DEVERR_BAD_LENGTH : HYB_DEVERR_BAD_BLOCK);
  const int lo = WINDOW ? window_lo(n, window) : 0;   // keys [lo, n)
  const int nblk = (n + kBlockSize - 1) / kBlockSize;
  const int nsplit = PREFILL ? 1 : decode_splits(n, WINDOW ? window : 0);
  if (split >= nsplit) return;
  const int blk_begin = lo / kBlockSize + split * kBPS;
  const int blk_end = PREFILL ? nblk : min(nblk, blk_begin + kBPS);

  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* btrow = bt + (int64_t)b * MB;
  const int sub_mask = (1 << rsh) - 1;
  const int64_t head_off = (int64_t)h * (kBlockSize << rsh) * D;
  const int64_t blk_stride = (int64_t)H * (kBlockSize << rsh) * D;
  constexpr int kRowChunks = D * (int)sizeof(T) / 16;   // 16-byte pieces of one K or V row

  // Append fused into the decode: the last split of (r, h) stores this step's k/v row at
  // slot_map[r]; when that slot is the one of position n - 1 (the normal decode step), the
  // warp that loads that position's tile also patches the row into shared memory, so the
  // attention sees exactly what an append followed by the decode would.
  int patch_sub = -1;                      // 16-token sub-tile holding position n - 1, if patched
  int64_t app_slot = -1;                   // where this step's row goes (-1: nowhere)
  if (!PREFILL && k_new && split == nsplit - 1) {
    const int bsz = kBlockSize << rsh;
    int64_t slot = -1;
    if (slot_map) {
      slot = slot_map[r];
    } else if (n >= 1) {                   // no slot mapping: position n - 1 through the table
      const int pb = btrow[((n - 1) / kBlockSize) >> rsh];
      if (pb >= 0 && pb < NB) slot = (int64_t)pb * bsz + (n - 1) % bsz;
    }
    if (slot >= (int64_t)NB * bsz) {
      if (threadIdx.x == 0) flag(status, HYB_DEVERR_BAD_SLOT);
      slot = -1;
    }
    if (slot >= 0) {
      app_slot = slot;                     // stored below, once the inputs may be read
      if (n >= 1) {
        const int s_last = (n - 1) / kBlockSize;
        const int pb = btrow[s_last >> rsh];
        if (pb >= 0 && pb < NB && slot == (int64_t)pb * bsz + (n - 1) % bsz) patch_sub = s_last;
      }
    }
  }

  uint8_t* ring = smem + (size_t)warp * kNST * 2 * TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)kNW * kNST * 2 * TILE) + warp * kNST;
  float* red_acc = reinterpret_cast<float*>(smem + (size_t)kNW * kNST * 2 * TILE + kNW * kNST * 8);
  float* red_ml = red_acc + kNW * D;

  const int c = lane % LPR, rr = lane / LPR;
  const int first = blk_begin + warp;   // this warp's logical blocks: first + i*kNW
  const int ntiles = first < blk_end ? (blk_end - first + kNW - 1) / kNW : 0;
  // 16-token sub-tile s lives in block btrow[s >> rsh], rows (s & sub_mask) * 16 onwards

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kNST; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  auto issue = [&](int i) {              // lane 0 only
    const int sub = first + i * kNW;
    const int pb = btrow[sub >> rsh];
    if (pb < 0 || pb >= NB) return;      // the consumer flags and skips it
    const int st = i % kNST;
    uint8_t* dst = ring + st * 2 * TILE;
    const int64_t off = pb * blk_stride + head_off + (int64_t)(sub & sub_mask) * kBlockSize * D;
    mbar_expect_tx(&bars[st], 2 * TILE);
    bulk_g2s(dst, kc + off, TILE, &bars[st]);
    bulk_g2s(dst + TILE, vc + off, TILE, &bars[st]);
  };
  if (lane == 0)
    for (int i = 0; i < min(kNST, ntiles); ++i) issue(i);

  // The next kernel may launch now: it waits for this one to complete before reading what
  // this one writes. (A kernel that is not early has already waited, so whatever an early
  // kernel launched after it reads before its own wait was complete before this launch.)
  pdl_trigger();
  if (app_slot >= 0 && warp == kNW - 1) {  // the append: this step's row into its slot
    const int bsz = kBlockSize << rsh;
    const int64_t blk = app_slot / bsz, off = app_slot - blk * bsz;
    const int64_t dst = ((blk * H + h) * bsz + off) * D;
    const int64_t src = ((int64_t)r * H + h) * D;
    for (int e = lane; e < kRowChunks; e += 32) {
      reinterpret_cast<uint4*>(kc + dst)[e] = reinterpret_cast<const uint4*>(k_new + src)[e];
      reinterpret_cast<uint4*>(vc + dst)[e] = reinterpret_cast<const uint4*>(v_new + src)[e];
    }
  }
  float qf[VEC];
  {
    const uint4 u = *reinterpret_cast<const uint4*>(q + ((int64_t)r * H + h) * D + c * VEC);
    E::unpack(u, qf);
#pragma unroll
    for (int e = 0; e < VEC; ++e) qf[e] *= scale_log2;
  }

  float m = -INFINITY, l = 0.f, acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  uint32_t phase = 0;
  int failed_at = -1;

  for (int i = 0; i < ntiles; ++i) {
    const int st = i % kNST;
    const int pb = btrow[(first + i * kNW) >> rsh];
    if (pb < 0 || pb >= NB) {
      if (lane == 0) flag(status, HYB_DEVERR_BAD_BLOCK);
    } else {
      if (!mbar_wait(&bars[st], (phase >> st) & 1u)) {
        failed_at = i;
        break;
      }
      phase ^= 1u << st;
      const T* Ks = reinterpret_cast<const T*>(ring + st * 2 * TILE);
      const T* Vs = reinterpret_cast<const T*>(ring + st * 2 * TILE + TILE);
      const int tok0 = (first + i * kNW) * kBlockSize;
      if (first + i * kNW == patch_sub) {  // this step's row, straight from the inputs
        const int row = (n - 1) % kBlockSize;
        const int64_t src = ((int64_t)r * H + h) * D;
        uint4* kd = reinterpret_cast<uint4*>(ring + st * 2 * TILE) + row * kRowChunks;
        uint4* vd = reinterpret_cast<uint4*>(ring + st * 2 * TILE + TILE) + row * kRowChunks;
        for (int e = lane; e < kRowChunks; e += 32) {
          kd[e] = reinterpret_cast<const uint4*>(k_new + src)[e];
          vd[e] = reinterpret_cast<const uint4*>(v_new + src)[e];
        }
        __syncwarp();
      }
      float s[ITER];
      float mt = -INFINITY;
#pragma unroll
      for (int it = 0; it < ITER; ++it) {
        const int tk = rr + it * TPI;
        float kf[VEC];
        E::unpack(*reinterpret_cast<const uint4*>(Ks + tk * D + c * VEC), kf);
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) d = fmaf(qf[e], kf[e], d);
#pragma unroll
        for (int o = LPR / 2; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        s[it] = (tok0 + tk < n && (!WINDOW || tok0 + tk >= lo)) ? d : -INFINITY;
        mt = fmaxf(mt, s[it]);
      }
#pragma unroll
      for (int o = LPR; o < 32; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      const float m_new = fmaxf(m, mt);  // finite: every tile holds a key in [lo, n)
      const float alpha = fast_exp2(m - m_new);
      float ls = 0.f;
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[e] *= alpha;
#pragma unroll
      for (int it = 0; it < ITER; ++it) {
        const int tk = rr + it * TPI;
        const float p = fast_exp2(s[it] - m_new);
        ls += p;
        if (tok0 + tk < n && (!WINDOW || tok0 + tk >= lo)) {   // others may hold NaN
          float vf[VEC];
          E::unpack(*reinterpret_cast<const uint4*>(Vs + tk * D + c * VEC), vf);
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[e] = fmaf(p, vf[e], acc[e]);
        }
      }
#pragma unroll
      for (int o = LPR; o < 32; o <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
      l = l * alpha + ls;
      m = m_new;
    }
    __syncwarp();
    if (lane == 0 && i + kNST < ntiles) issue(i + kNST);
  }

  if (failed_at >= 0) {
    // A wait expired: report, then let the copies still in flight land before exiting.
    if (lane == 0) {
      flag(status, HYB_DEVERR_TIMEOUT);
      for (int j = failed_at; j < min(failed_at + kNST, ntiles); ++j) {
        const int pb = btrow[(first + j * kNW) >> rsh];
        if (pb >= 0 && pb < NB) {
          const int st = j % kNST;
          mbar_wait(&bars[st], (phase >> st) & 1u, 100000000ull);
          phase ^= 1u << st;
        }
      }
    }
    __syncwarp();
    m = -INFINITY; l = 0.f;
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  }

  // merge the token sub-rows of the warp (lanes with the same c)
#pragma unroll
  for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
  if (lane < LPR)
#pragma unroll
    for (int e = 0; e < VEC; ++e) red_acc[warp * D + c * VEC + e] = acc[e];
  if (lane == 0) {
    red_ml[2 * warp] = m;
    red_ml[2 * warp + 1] = l;
  }
  __syncthreads();
  // Early: the previous kernel (the previous layer's split combine) may still be reading the
  // split workspace; every write comes after it has completed, and so does this kernel's end
  // (so the next kernel's wait covers every earlier kernel of the dispatch).
  if (early) pdl_wait();

  for (int t = threadIdx.x; t < D; t += kNW * 32) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kNW; ++w) M = fmaxf(M, red_ml[2 * w]);
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kNW; ++w) {
        const float sc = fast_exp2(red_ml[2 * w] - M);
        L = fmaf(red_ml[2 * w + 1], sc, L);
        A = fmaf(red_acc[w * D + t], sc, A);
      }
    }
    const int64_t rh = (int64_t)r * H + h;
    if (nsplit == 1) {
      E::store(out + rh * D + t, L > 0.f ? A / L : 0.f);
    } else {
      ws_acc[(rh * max_splits + split) * D + t] = A;
      if (t == 0) ws_ml[rh * max_splits + split] = make_float2(M, L);
    }
  }
}

// Split sums of one output element for a row with at most NS splits: every (m, l) pair and
// partial sum is loaded before the maximum is taken, so they take one round trip.
template <int NS, int D>
__device__ __forceinline__ void combine_few(const float2* __restrict__ ml,
                                            const float* __restrict__ acc, int nsplit, int t,
                                            float& L, float& A) {
  float2 v[NS];
  float a[NS];
#pragma unroll
  for (int u = 0; u < NS; ++u) {
    v[u] = u < nsplit ? ml[u] : make_float2(-INFINITY, 0.f);
    a[u] = u < nsplit ? acc[(int64_t)u * D + t] : 0.f;
  }
  float M = v[0].x;
#pragma unroll
  for (int u = 1; u < NS; ++u) M = fmaxf(M, v[u].x);
  if (M == -INFINITY) return;
#pragma unroll
  for (int u = 0; u < NS; ++u) {
    if (u < nsplit) {
      const float sc = fast_exp2(v[u].x - M);
      L = fmaf(v[u].y, sc, L);
      A = fmaf(a[u], sc, A);
    }
  }
}

// Merges the splits of one (request, head): out = sum_s 2^(m_s-M) acc_s / sum_s 2^(m_s-M) l_s.
// Every thread takes the max M itself from the (m, l) pairs (the same addresses for all
// threads, so one broadcast load each): no block reduction, and with at most 16 splits the
// pairs and the partial sums are all loaded in one round trip. The sums keep split order,
// so results do not depend on the CTA shape or on which branch a row takes.
template <typename T, int D>
__global__ void __launch_bounds__(128)
decode_combine_kernel(T* __restrict__ out, const int32_t* __restrict__ seq_lens, int H, int MBt,
                      int max_len, int window, int max_splits, const float* __restrict__ ws_acc,
                      const float2* __restrict__ ws_ml) {
  // seq_lens was read by the decode launched just before, after its own wait: rows with one
  // split leave before waiting, and the next kernel may launch at once (it waits for this
  // one to complete before reading anything it writes)
  const int r = blockIdx.x, h = blockIdx.y;
  const int n = clamp_len(seq_lens[r], max_len, MBt);
  const int nsplit = decode_splits(n, window);
  if (nsplit <= 1) return;
  pdl_trigger();
  pdl_wait();
  const int64_t rh = (int64_t)r * H + h;
  const float2* ml = ws_ml + rh * max_splits;
  const float* acc = ws_acc + rh * max_splits * D;
  for (int t = threadIdx.x; t < D; t += blockDim.x) {
    float L = 0.f, A = 0.f;
    if (nsplit <= 8) {
      combine_few<8, D>(ml, acc, nsplit, t, L, A);
    } else if (nsplit <= 16) {
      combine_few<16, D>(ml, acc, nsplit, t, L, A);
    } else {
      // long rows: 32 splits' loads in flight per round (the sums keep split order)
      constexpr int kR = 32;
      float M = -INFINITY;
      int s = 0;
      for (; s + kR <= nsplit; s += kR) {
        float m[kR];
#pragma unroll
        for (int u = 0; u < kR; ++u) m[u] = ml[s + u].x;
#pragma unroll
        for (int u = 0; u < kR; ++u) M = fmaxf(M, m[u]);
      }
      for (; s < nsplit; ++s) M = fmaxf(M, ml[s].x);
      if (M != -INFINITY) {
        s = 0;
        for (; s + kR <= nsplit; s += kR) {
          float2 v[kR];
          float a[kR];
#pragma unroll
          for (int u = 0; u < kR; ++u) {
            v[u] = ml[s + u];
            a[u] = acc[(int64_t)(s + u) * D + t];
          }
#pragma unroll
          for (int u = 0; u < kR; ++u) {
            const float sc = fast_exp2(v[u].x - M);
            L = fmaf(v[u].y, sc, L);
            A = fmaf(a[u], sc, A);
          }
        }
        for (; s < nsplit; ++s) {
          const float2 v = ml[s];
          const float sc = fast_exp2(v.x - M);
          L = fmaf(v.y, sc, L);
          A = fmaf(acc[(int64_t)s * D + t], sc, A);
        }
      }
    }
    Elt<T>::store(out + rh * D + t, L > 0.f ? A / L : 0.f);
  }
}

template <typename T, int D>
cudaError_t launch_typed(void* out, const void* q, const void* kc, const void* vc,
                         const int32_t* bt, const int32_t* seq_lens, const int32_t* cu,
                         const int32_t* ctx, int R, int max_q, int H, int NB, int MB,
                         int bs, int max_len, float scale, int window, const DecodePlan& plan,
                         void* ws, unsigned* status, cudaStream_t s, const DecodeAppend* app,
                         bool early) {
  using Sh = DecodeShape<T, D>;
  const bool prefill = cu != nullptr, win = window > 0;
  using K = void (*)(T*, const T*, T*, T*, const int32_t*, const int32_t*, const int32_t*,
                     const int32_t*, int, int, int, int, int, int, float, int, int, float*,
                     float2*, const T*, const T*, const int64_t*, int, unsigned*);
  const int rsh = log2_int(bs / kBlockSize);
  const K kern = prefill ? (win ? paged_decode_kernel<T, D, true, true>
                                : paged_decode_kernel<T, D, true, false>)
                         : (win ? paged_decode_kernel<T, D, false, true>
                                : paged_decode_kernel<T, D, false, false>);
  cudaError_t e = set_smem((const void*)kern, Sh::SMEM);
  if (e != cudaSuccess) return e;
  const int max_splits = prefill ? 1 : plan.max_splits;
  float* ws_acc = static_cast<float*>(ws);
  float2* ws_ml = reinterpret_cast<float2*>(
      static_cast<char*>(ws) + (size_t)R * H * max_splits * D * sizeof(float));
  // Decode CTAs start in linear order over (split, row, head), the split index fastest: a
  // row's splits are dispatched together, so in a batch of mixed lengths the splits of the
  // long rows do not wait behind a plane of (mostly empty) later splits and run alone at the
  // end. (Measured on the 32-layer step: 2.66 ms against 2.72 ms with the split slowest.)
  const dim3 grid = prefill ? dim3(R * max_q, H, 1) : dim3(max_splits, R, H);
  const float scale_log2 = scale * 1.4426950408889634f;
  const bool fused = app != nullptr && !prefill;
  e = launch_pdl(kern, grid, dim3(kNW * 32), Sh::SMEM, s, (T*)out, (const T*)q, (T*)kc, (T*)vc,
                 bt, seq_lens, cu, ctx, max_q, H, NB, MB, rsh, max_len, scale_log2, window,
                 max_splits, ws_acc, ws_ml, fused ? (const T*)app->k : (const T*)nullptr,
                 fused ? (const T*)app->v : (const T*)nullptr,
                 fused ? app->slot : (const int64_t*)nullptr, (early && !prefill) ? 1 : 0, status);
  count_launch();
  if (e != cudaSuccess || max_splits == 1) return e;
  e = launch_pdl(decode_combine_kernel<T, D>, dim3(R, H), dim3(128), 0, s, (T*)out, seq_lens, H,
                 MB << rsh, max_len, window, max_splits, (const float*)ws_acc,
                 (const float2*)ws_ml);
  count_launch();
  return e;
}

}  // namespace

DecodePlan plan_decode(int B, int H, int D, int max_seq_len, int window) {
  DecodePlan p;
  p.blocks_per_split = kBPS;
  int nblk = (std::max(max_seq_len, 0) + kBlockSize - 1) / kBlockSize;
  // `window` keys starting anywhere inside a block touch at most (window + 14) / 16 + 1 blocks
  if (window > 0) nblk = std::min(nblk, (window + kBlockSize - 2) / kBlockSize + 1);
  p.max_splits = std::max(1, (nblk + kBPS - 1) / kBPS);
  p.ws_bytes = p.max_splits > 1 ? (size_t)B * H * p.max_splits * ((size_t)D * 4 + 8) : 0;
  return p;
}

bool decode_supported(int dtype, int D) {
  if (dtype == HYB_BF16) return D == 16 || D == 32 || D == 64 || D == 128 || D == 256;
  if (dtype == HYB_F32) return D == 16 || D == 32 || D == 64 || D == 128;
  return false;
}

cudaError_t launch_paged_decode(void* out, const void* q, const void* kc, const void* vc,
                                const int32_t* bt, const int32_t* seq_lens, const int32_t* cu,
                                const int32_t* ctx, int R, int max_q, int H, int D, int dtype,
                                int NB, int MB, int bs, int max_len, float scale, int window,
                                const DecodePlan& plan, void* ws, unsigned* status,
                                cudaStream_t s, const DecodeAppend* app, bool early) {
  if (R == 0 || (cu && max_q == 0)) return cudaSuccess;
#define HYB_DEC(T, DD)                                                                       \
  if (D == DD)                                                                               \
    return launch_typed<T, DD>(out, q, kc, vc, bt, seq_lens, cu, ctx, R, max_q, H, NB, MB, bs, \
                               max_len, scale, window, plan, ws, status, s, app, early);
  if (dtype == HYB_BF16) {
    HYB_DEC(__nv_bfloat16, 16)
    HYB_DEC(__nv_bfloat16, 32)
    HYB_DEC(__nv_bfloat16, 64)
    HYB_DEC(__nv_bfloat16, 128)
    HYB_DEC(__nv_bfloat16, 256)
  } else {
    HYB_DEC(float, 16)
    HYB_DEC(float, 32)
    HYB_DEC(float, 64)
    HYB_DEC(float, 128)
  }
#undef HYB_DEC
  return cudaErrorInvalidValue;
}

}  // namespace hyb
