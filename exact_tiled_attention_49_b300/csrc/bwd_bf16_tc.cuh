// bwd_bf16_tc.cuh -- attention backward (dQ, dK, dV) on the tensor cores, bf16
// or fp16 (kF16) inputs and gradients.
//
// The chain rule through the softmax ("Hands-on build guide:
// FlashAttention-style tiled attention kernel in pure NumPy", Roadmap:
// gradient through attention), with the weights recomputed on chip from
// the forward's per-row log-sum-exp instead of being stored ("Self-Attention:
// Implementation, Complexity, and Efficient Variants", FlashAttention: the
// backward pass recomputes the attention matrix on chip):
//
//   P  = exp(scale * Q K^T - LSE)      (0 on hidden keys and empty rows)
//   dP = dO V^T,  delta = rowsum(dO * O),  dS = P * (dP - delta)
//   dQ = scale * dS K,  dK = scale * dS^T Q,  dV = P^T dO
//
// Three kernels, no atomics (results do not depend on scheduling):
//   bwd_delta_kernel       delta = rowsum(dO * O) in fp32 (CUDA cores).
//   bwd_dq_kernel<D>       one CTA per (128-row query tile, head, batch):
//                          S = Q K_j^T and dP = dO V_j^T into TMEM, dS in
//                          the softmax warps, dQ += dS K_j (A = dS from TMEM).
//   bwd_dkdv_kernel<D>     one CTA per (128-key tile, kv head, batch); it
//                          walks the query tiles of every query head of its
//                          group: S^T = K Q_i^T and dP^T = V dO_i^T (so that
//                          thread r owns key r), P^T and dS^T in the softmax
//                          warps, dV += P^T dO_i and dK += dS^T Q_i.
// S and dP are computed in both kernels: two extra products buy freedom from
// atomics.  Warp roles as in the forward: warps 0-3 elementwise (thread r =
// TMEM lane r), warp 4 TMA producer, warp 5 MMA issuer (converged, one
// elected lane issues).  Every mbarrier wait is bounded.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace attn {
namespace tcbwd {

constexpr int kBM = 128;       // rows of an MMA tile (= TMEM lanes)
constexpr int kThreads = 192;  // 4 elementwise warps + load warp + MMA warp
constexpr int kLoadWarp = 4;
constexpr int kMmaWarp = 5;

struct Params {
  const void* o;            // [B,Hq,T,D] bf16 (delta kernel)
  const void* dout;         // [B,Hq,T,D] bf16 (delta kernel)
  const float* lse;         // [B,Hq,T]
  float* delta;             // [B,Hq,T] workspace
  void* dq;                 // [B,Hq,T,D] bf16
  void* dk;                 // [B,Hkv,S,D] bf16
  void* dv;                 // [B,Hkv,S,D] bf16
  const int32_t* key_lens;  // [B] or null
  const int32_t* q_pos;     // [B] or null (S - T)
  int B, Hq, Hkv, T, S, D;
  int causal;
  int n_qtiles, n_ktiles;
  float scale;              // softmax scale
  float scale_log2;         // scale * log2(e)
};

__device__ __forceinline__ int key_bound(const Params& p, int b) {
  return p.key_lens != nullptr ? min(max(p.key_lens[b], 0), p.S) : p.S;
}

// Key position of query row 0 of sequence b (see the forward kernel).
__device__ __forceinline__ int q_offset(const Params& p, int b) {
  return p.q_pos != nullptr ? min(max(p.q_pos[b], -(p.T + 256)), p.S) : p.S - p.T;
}

// ------------------------------------------------------------ delta pass
// delta[row] = sum_d dO[row,d] * O[row,d] in fp32.  A row is D / 8 lanes of
// one 16-byte vector each (16 lanes at D = 128, 8 at D = 64), so a warp
// takes 32 / (D / 8) rows at a time with every lane loading; the lanes of a
// row add their partial dot products with xor shuffles inside their group.
template <bool kF16>
__global__ void __launch_bounds__(256) bwd_delta_kernel(Params p, long long rows) {
  const int lpr = p.D / 8;   // lanes per row
  const int rpw = 32 / lpr;  // rows per warp step
  const long long warp_id = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = ((long long)gridDim.x * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / lpr, c = lane - sub * lpr;
  for (long long r0 = warp_id * rpw; r0 < rows; r0 += n_warps * rpw) {
    const long long r = r0 + sub;
    float acc = 0.f;
    if (r < rows) {
      const uint4 a = reinterpret_cast<const uint4*>(p.o)[r * lpr + c];
      const uint4 g = reinterpret_cast<const uint4*>(p.dout)[r * lpr + c];
      acc = fmaf(elem_lo<kF16>(a.x), elem_lo<kF16>(g.x), acc);
      acc = fmaf(elem_hi<kF16>(a.x), elem_hi<kF16>(g.x), acc);
      acc = fmaf(elem_lo<kF16>(a.y), elem_lo<kF16>(g.y), acc);
      acc = fmaf(elem_hi<kF16>(a.y), elem_hi<kF16>(g.y), acc);
      acc = fmaf(elem_lo<kF16>(a.z), elem_lo<kF16>(g.z), acc);
      acc = fmaf(elem_hi<kF16>(a.z), elem_hi<kF16>(g.z), acc);
      acc = fmaf(elem_lo<kF16>(a.w), elem_lo<kF16>(g.w), acc);
      acc = fmaf(elem_hi<kF16>(a.w), elem_hi<kF16>(g.w), acc);
    }
    for (int off = lpr >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (c == 0 && r < rows) p.delta[r] = acc;
  }
}

// ---------------------------------------------------------- shared setup

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;
  static constexpr uint32_t kTileBytes = kBM * D * 2;       // one 128-row tile
  static constexpr uint32_t kChunkBytes = kBM * 128;        // 128 rows x 128 B
  static constexpr int kStages = (D == 128) ? 2 : 4;        // streamed (X, Y) tile pairs
  static constexpr uint32_t kOffFixed = 0;                  // two resident tiles
  static constexpr uint32_t kOffRing = 2 * kTileBytes;
  static constexpr uint32_t kOffStats = kOffRing + kStages * 2 * kTileBytes;
  // dK/dV kernel: per elementwise warp, the 128 LSE and delta values of the
  // current query tile (4 warps x 2 x 128 floats)
  static constexpr uint32_t kOffBars = kOffStats + 4 * 2 * kBM * 4;
  // barriers: fixed_full, ring_full[kStages], ring_empty[kStages], mm[2]
  // (S and dP of a 64-column half done), pp[2] (that half's packed P / dS
  // in TMEM), acc_full, drain, tail (dQ kernel: the K/V tile that straddles
  // the valid key length)
  static constexpr int kNumBars = 1 + 2 * kStages + 7;
  static constexpr uint32_t kOffMisc = kOffBars + 8 * kNumBars;
  static constexpr uint32_t kBytes = kOffMisc + 16;
  static constexpr size_t kSmemAlloc = kBytes + 1024;
};

// Both kernels split every 128x128 product tile into two 64-column halves
// with their own TMEM columns: half h holds S (or S^T) at 128h and dP (or
// dP^T) at 128h + 64.  The MMA warp issues S/dP of one half while the
// elementwise warps turn the other half into packed bf16 P / dS (written
// back over the first 32 columns of S and dP), so the tensor core and the
// CUDA cores overlap:
//
//   MMA:  SdP(u,0) SdP(u,1) | acc(u,0) SdP(u+1,0) | acc(u,1) SdP(u+1,1) | ...
//   ALU:        half(u,0)   |   half(u,1)         |   half(u+1,0)       | ...
//
// The accumulating products read a half's packed operand before the next
// S/dP of that half overwrites its columns: tcgen05.mma operations issued
// by one thread execute in order.
constexpr int kHalf = 64;
__device__ __forceinline__ constexpr uint32_t col_s(int h) { return 128u * h; }
__device__ __forceinline__ constexpr uint32_t col_dp(int h) { return 128u * h + 64u; }
constexpr uint32_t kColAcc = 256;

// ------------------------------------------------------------- dQ kernel
//
// Grid: x = (batch, query head), y = query tile, heaviest causal tiles first
// (y = 0 is the last query tile).  TMEM: S/dP halves at 0..255, dQ at 256.
template <int D, bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, Params p) {
  using C = Cfg<D>;
  constexpr uint32_t kColDQ = kColAcc, kTmemCols = 512;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t s_q = sbase + C::kOffFixed, s_do = s_q + C::kTileBytes;
  const uint32_t s_ring = sbase + C::kOffRing;  // stage s: K at 2s, V at 2s+1
  const uint32_t bars = sbase + C::kOffBars;
  const uint32_t bar_fixed = bars;
  auto bar_full = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_empty = [&](int s) { return bars + 8u * (1 + C::kStages + s); };
  const uint32_t bar_mm0 = bars + 8u * (1 + 2 * C::kStages);  // mm[h] = bar_mm0 + 8h
  const uint32_t bar_pp0 = bar_mm0 + 16;                       // pp[h] = bar_pp0 + 8h
  const uint32_t bar_acc = bar_pp0 + 16, bar_drain = bar_acc + 8, bar_tail = bar_drain + 8;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = p.n_qtiles - 1 - (int)blockIdx.y;
  const int b = (int)blockIdx.x / p.Hq, h = (int)blockIdx.x % p.Hq;
  const int g = h / (p.Hq / p.Hkv);
  const int q0 = qt * kBM;
  const int L = key_bound(p, b);
  const int off = q_offset(p, b);
  // key tiles this query tile visits
  int n = 0;
  if (q0 < p.T && q0 + off < L) {
    const int kv_end = p.causal ? min(L, q0 + kBM + off) : L;
    n = kv_end > 0 ? (kv_end + kBM - 1) / kBM : 0;
  }

  if (threadIdx.x == 0) {
    mbar_init(bar_fixed, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_mm0, 1);
    mbar_init(bar_mm0 + 8, 1);
    mbar_init(bar_pp0, 4 * 32);
    mbar_init(bar_pp0 + 8, 4 * 32);
    mbar_init(bar_acc, 1);
    mbar_init(bar_drain, 1);
    mbar_init(bar_tail, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int bh_q = b * p.Hq + h, bh_kv = b * p.Hkv + g;

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop; lane 0 issues the copies.  The K/V tile
    // that straddles the valid key length L lands on a private barrier and
    // its rows at or past L are zeroed before the tile is released: dS is 0
    // there, but dQ += dS K would turn 0 * NaN into NaN.
    if (n > 0) {
      if (lane == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_do);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        mbar_arrive_expect_tx(bar_fixed, 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(s_q + c * C::kChunkBytes, &tm_q, bar_fixed, c * 64, q0, bh_q);
          tma_load_3d(s_do + c * C::kChunkBytes, &tm_do, bar_fixed, c * 64, q0, bh_q);
        }
      }
      const int j_tail = (L < p.S && (L & (kBM - 1)) != 0) ? L / kBM : -1;
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        const int s = j % C::kStages;
        if (j >= C::kStages &&
            !__all_sync(0xffffffffu,
                        mbar_wait(bar_empty(s), ((j / C::kStages) - 1) & 1, 1, abort_flag)))
          break;
        const uint32_t dk = s_ring + 2 * s * C::kTileBytes, dv = dk + C::kTileBytes;
        const bool tail = j == j_tail;
        const uint32_t bar_land = tail ? bar_tail : bar_full(s);
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_land, 2 * C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c) {
            tma_load_3d(dk + c * C::kChunkBytes, &tm_k, bar_land, c * 64, j * kBM, bh_kv);
            tma_load_3d(dv + c * C::kChunkBytes, &tm_v, bar_land, c * 64, j * kBM, bh_kv);
          }
        }
        issued = j + 1;
        if (tail) {
          if (!__all_sync(0xffffffffu, mbar_wait(bar_tail, 0, 1, abort_flag))) break;
          const int r0 = L & (kBM - 1);
          for (int idx = r0 * 8 + lane; idx < kBM * 8; idx += 32)
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
              st_shared_zero16(dk + c * C::kChunkBytes + idx * 16);
              st_shared_zero16(dv + c * C::kChunkBytes + idx * 16);
            }
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_full(s));
        }
      }
      // drain: every issued copy lands before exit
      mbar_wait(bar_fixed, 0, 2);
      for (int j = max(0, issued - C::kStages); j < issued; ++j)
        if (j != j_tail) mbar_wait(bar_full(j % C::kStages), (j / C::kStages) & 1, 2);
      if (j_tail >= 0 && j_tail < issued) mbar_wait(bar_tail, 0, 2);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc_s = idesc_f16kind(kBM, kHalf, false, false, kF16);  // M=128, N=64, K-major
    constexpr uint32_t idesc_ts = idesc_f16kind(kBM, D, false, true, kF16);      // B MN-major, N = D
    const uint64_t dq_a = sdesc_sw128(s_q, 16, 1024), ddo_a = sdesc_sw128(s_do, 16, 1024);
    const uint64_t dk0 = sdesc_sw128(s_ring, 16, 1024);
    const uint64_t dkmn0 = sdesc_sw128(s_ring, C::kChunkBytes, 1024);
    bool ok = n > 0 && __all_sync(0xffffffffu, mbar_wait(bar_fixed, 0, 3, abort_flag));
    // S_h = Q K_j[64h, 64h + 64)^T and dP_h = dO V_j[64h, 64h + 64)^T: the
    // B operand starts 64 rows (8 swizzle atoms) into each 128-row chunk.
    auto issue_sdp = [&](int s, int hh) {
      const uint64_t rows = (uint64_t)((hh * kHalf * 128) >> 4);
      const uint64_t dk = dk0 + (uint64_t)((2 * s * C::kTileBytes) >> 4) + rows;
      const uint64_t dv = dk0 + (uint64_t)(((2 * s + 1) * C::kTileBytes) >> 4) + rows;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ko = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
        umma_ss_elect(tmem + col_s(hh), dq_a + ko, dk + ko, idesc_s, kk > 0);
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ko = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
        umma_ss_elect(tmem + col_dp(hh), ddo_a + ko, dv + ko, idesc_s, kk > 0);
      }
      umma_commit_elect(bar_mm0 + 8u * hh);
    };
    // dQ += dS_h K_j[64h, 64h + 64): A = packed dS_h in TMEM, K = 64 keys
    auto issue_dq = [&](int s, int hh, bool first) {
      const uint64_t dkmn = dkmn0 + (uint64_t)((2 * s * C::kTileBytes) >> 4) + (uint64_t)(hh * 4 * 128);
#pragma unroll
      for (int kk = 0; kk < kHalf / 16; ++kk)
        umma_ts_elect(tmem + kColDQ, tmem + col_s(hh) + kk * 8, dkmn + (uint64_t)(kk * 128),
                      idesc_ts, (!first || kk > 0) ? 1u : 0u);
    };
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_full(0), 0, 4, abort_flag));
      if (ok) {
        tc_fence_after();
        issue_sdp(0, 0);
        issue_sdp(0, 1);
      }
    }
    for (int j = 0; ok && j < n; ++j) {
      const int s = j % C::kStages, s1 = (j + 1) % C::kStages;
      const bool more = j + 1 < n;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_pp0, j & 1, 5, abort_flag)))) break;
      tc_fence_after();
      issue_dq(s, 0, j == 0);
      if (more) {
        if (!(ok = __all_sync(0xffffffffu,
                              mbar_wait(bar_full(s1), ((j + 1) / C::kStages) & 1, 4, abort_flag))))
          break;
        tc_fence_after();
        issue_sdp(s1, 0);
      }
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_pp0 + 8, j & 1, 5, abort_flag)))) break;
      tc_fence_after();
      issue_dq(s, 1, false);
      umma_commit_elect(bar_empty(s));
      if (more) issue_sdp(s1, 1);
      else umma_commit_elect(bar_acc);
    }
    umma_commit_elect(bar_drain);
    mbar_wait(bar_drain, 0, 6);
    __syncwarp();
  } else {
    // --------------------------------------------------------- elementwise
    const int r = threadIdx.x;  // query row within the tile = TMEM lane
    const int i = q0 + r;
    const int pos = i + off;
    const bool row_ok = (i < p.T) && (pos < L);
    const int lim = !row_ok ? 0 : (p.causal ? min(L, pos + 1) : L);  // visible keys [0, lim)
    const int lim_warp = __reduce_min_sync(0xffffffffu, lim);
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const size_t row = ((size_t)b * p.Hq + h) * p.T + i;
    const float lse2 = row_ok ? p.lse[row] * 1.4426950408889634f : 0.f;
    const float dlt = row_ok ? p.delta[row] : 0.f;
    const float2 sl2x2 = make_float2(p.scale_log2, p.scale_log2);
    const float2 nl2 = make_float2(-lse2, -lse2);
    const float2 ndl2 = make_float2(-dlt, -dlt);
    bool ok = true;
    for (int j = 0; ok && j < n; ++j) {
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar_mm0 + 8u * hh, j & 1, 7, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const int kb = j * kBM + hh * kHalf;  // first key of the half
        // Every key of the half visible to every row of the warp: no masks.
        const bool dense = kb + kHalf <= lim_warp;
        // 32 columns at a time: P = exp2(s * scale*log2e - lse*log2e) on
        // visible keys, dS = P (dP - delta), packed to bf16 over the first
        // 32 columns of the half's S (chunk c goes to columns 16c.., all of
        // which have been read by then).
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t sr[32], dp[32];
          tmem_ld32(lane_base + col_s(hh) + 32 * c, sr);
          tmem_ld32(lane_base + col_dp(hh) + 32 * c, dp);
          tmem_wait_ld32(sr);
          tmem_wait_ld32(dp);
          uint32_t pk[16];
          if (dense) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                          sl2x2, nl2);
              const float2 pe = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              const float2 d = __fadd2_rn(make_float2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])),
                                          ndl2);
              const float2 ds = __fmul2_rn(pe, d);
              pk[e >> 1] = pack2<kF16>(ds.x, ds.y);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const int kj = kb + 32 * c + e;
              // selects, not products: hidden entries may hold NaN (keys past
              // the valid length), and 0 * NaN would be NaN
              const float p0 = ex2_approx(fmaf(__uint_as_float(sr[e]), sl2x2.x, -lse2));
              const float p1 = ex2_approx(fmaf(__uint_as_float(sr[e + 1]), sl2x2.x, -lse2));
              const float d0 = (kj < lim) ? p0 * (__uint_as_float(dp[e]) - dlt) : 0.f;
              const float d1 = (kj + 1 < lim) ? p1 * (__uint_as_float(dp[e + 1]) - dlt) : 0.f;
              pk[e >> 1] = pack2<kF16>(d0, d1);
            }
          }
          tmem_st16(lane_base + col_s(hh) + 16 * c, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_pp0 + 8u * hh);
      }
    }
    // ------------------------------------------------------------ epilogue
    if (ok && n > 0) ok = __all_sync(0xffffffffu, mbar_wait(bar_acc, 0, 8, abort_flag));
    const bool has = ok && n > 0;  // warp-uniform
    if (has) tc_fence_after();
    const float sc = row_ok ? p.scale : 0.f;
    uint16_t* drow = reinterpret_cast<uint16_t*>(p.dq) + row * D;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t a[32];
      if (has) {
        tmem_ld32(lane_base + kColDQ + 32 * c, a);
        tmem_wait_ld32(a);
      }
      if (i < p.T) {
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          uint4 u = make_uint4(0, 0, 0, 0);
          if (has) {
            u.x = pack2<kF16>(__uint_as_float(a[8 * v4 + 0]) * sc, __uint_as_float(a[8 * v4 + 1]) * sc);
            u.y = pack2<kF16>(__uint_as_float(a[8 * v4 + 2]) * sc, __uint_as_float(a[8 * v4 + 3]) * sc);
            u.z = pack2<kF16>(__uint_as_float(a[8 * v4 + 4]) * sc, __uint_as_float(a[8 * v4 + 5]) * sc);
            u.w = pack2<kF16>(__uint_as_float(a[8 * v4 + 6]) * sc, __uint_as_float(a[8 * v4 + 7]) * sc);
          }
          reinterpret_cast<uint4*>(drow + 32 * c)[v4] = u;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ----------------------------------------------------------- dK/dV kernel
//
// Grid: x = (batch, kv head), y = key tile (the first key tiles are the
// heaviest under a causal mask).  TMEM: S^T/dP^T halves at 0..255 (a half =
// 64 query columns; P^T and dS^T packed over the first 32 columns of each),
// dV at 256, dK at 256 + D.
template <int D, bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, Params p) {
  using C = Cfg<D>;
  constexpr uint32_t kColDV = kColAcc, kColDK = kColAcc + D;
  constexpr uint32_t kTmemCols = 512;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t s_k = sbase + C::kOffFixed, s_v = s_k + C::kTileBytes;
  const uint32_t s_ring = sbase + C::kOffRing;  // stage s: Q at 2s, dO at 2s+1
  float* stats = reinterpret_cast<float*>(smem + C::kOffStats);
  const uint32_t bars = sbase + C::kOffBars;
  const uint32_t bar_fixed = bars;
  auto bar_full = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_empty = [&](int s) { return bars + 8u * (1 + C::kStages + s); };
  const uint32_t bar_mm0 = bars + 8u * (1 + 2 * C::kStages);
  const uint32_t bar_pp0 = bar_mm0 + 16;
  const uint32_t bar_acc = bar_pp0 + 16, bar_drain = bar_acc + 8;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kt = (int)blockIdx.y;
  const int b = (int)blockIdx.x / p.Hkv, g = (int)blockIdx.x % p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int k0 = kt * kBM;
  const int L = key_bound(p, b);
  const int off = q_offset(p, b);
  // Query tiles that see some key of this tile: rows i with pos = i + off in
  // [max(k0, 0) (causal), L) and i < T.
  int i_lo = 0, i_hi = 0;
  if (k0 < L) {
    i_lo = p.causal ? max(0, k0 - off) / kBM : 0;  // causal: rows with pos >= k0
    const int i_end = min(p.T, L - off);  // rows past this are padded
    i_hi = i_end > 0 ? (i_end + kBM - 1) / kBM : 0;
    if (i_hi < i_lo) i_hi = i_lo;
  }
  const int n_tiles_per_head = i_hi - i_lo;
  const int n = n_tiles_per_head * G;  // (query head, query tile) items

  if (threadIdx.x == 0) {
    mbar_init(bar_fixed, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_mm0, 1);
    mbar_init(bar_mm0 + 8, 1);
    mbar_init(bar_pp0, 4 * 32);
    mbar_init(bar_pp0 + 8, 4 * 32);
    mbar_init(bar_acc, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int bh_kv = b * p.Hkv + g;

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_do);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      mbar_arrive_expect_tx(bar_fixed, 2 * C::kTileBytes);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(s_k + c * C::kChunkBytes, &tm_k, bar_fixed, c * 64, k0, bh_kv);
        tma_load_3d(s_v + c * C::kChunkBytes, &tm_v, bar_fixed, c * 64, k0, bh_kv);
      }
      for (int u = 0; u < n; ++u) {
        const int s = u % C::kStages;
        if (u >= C::kStages && !mbar_wait(bar_empty(s), ((u / C::kStages) - 1) & 1, 1, abort_flag))
          break;
        const int hq = g * G + u / n_tiles_per_head;
        const int q0 = (i_lo + u % n_tiles_per_head) * kBM;
        const uint32_t dq_ = s_ring + 2 * s * C::kTileBytes, ddo = dq_ + C::kTileBytes;
        mbar_arrive_expect_tx(bar_full(s), 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(dq_ + c * C::kChunkBytes, &tm_q, bar_full(s), c * 64, q0, b * p.Hq + hq);
          tma_load_3d(ddo + c * C::kChunkBytes, &tm_do, bar_full(s), c * 64, q0, b * p.Hq + hq);
        }
      }
      mbar_wait(bar_fixed, 0, 2);
      for (int u = max(0, n - C::kStages); u < n; ++u)
        mbar_wait(bar_full(u % C::kStages), (u / C::kStages) & 1, 2);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc_s = idesc_f16kind(kBM, kHalf, false, false, kF16);
    constexpr uint32_t idesc_ts = idesc_f16kind(kBM, D, false, true, kF16);
    const uint64_t dk_a = sdesc_sw128(s_k, 16, 1024), dv_a = sdesc_sw128(s_v, 16, 1024);
    const uint64_t dr0 = sdesc_sw128(s_ring, 16, 1024);
    const uint64_t drmn0 = sdesc_sw128(s_ring, C::kChunkBytes, 1024);
    bool ok = n > 0 && __all_sync(0xffffffffu, mbar_wait(bar_fixed, 0, 3, abort_flag));
    // S^T_h = K Q[64h, 64h + 64)^T and dP^T_h = V dO[64h, 64h + 64)^T
    auto issue_sdp = [&](int s, int hh) {
      const uint64_t rows = (uint64_t)((hh * kHalf * 128) >> 4);
      const uint64_t dq_ = dr0 + (uint64_t)((2 * s * C::kTileBytes) >> 4) + rows;
      const uint64_t ddo = dr0 + (uint64_t)(((2 * s + 1) * C::kTileBytes) >> 4) + rows;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ko = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
        umma_ss_elect(tmem + col_s(hh), dk_a + ko, dq_ + ko, idesc_s, kk > 0);
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ko = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
        umma_ss_elect(tmem + col_dp(hh), dv_a + ko, ddo + ko, idesc_s, kk > 0);
      }
      umma_commit_elect(bar_mm0 + 8u * hh);
    };
    // dV += P^T_h dO[64h..] and dK += dS^T_h Q[64h..], K = 64 queries
    auto issue_acc = [&](int s, int hh, bool first) {
      const uint64_t half = (uint64_t)(hh * 4 * 128);
      const uint64_t dqmn = drmn0 + (uint64_t)((2 * s * C::kTileBytes) >> 4) + half;
      const uint64_t ddomn = drmn0 + (uint64_t)(((2 * s + 1) * C::kTileBytes) >> 4) + half;
#pragma unroll
      for (int kk = 0; kk < kHalf / 16; ++kk)
        umma_ts_elect(tmem + kColDV, tmem + col_s(hh) + kk * 8, ddomn + (uint64_t)(kk * 128),
                      idesc_ts, (!first || kk > 0) ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < kHalf / 16; ++kk)
        umma_ts_elect(tmem + kColDK, tmem + col_dp(hh) + kk * 8, dqmn + (uint64_t)(kk * 128),
                      idesc_ts, (!first || kk > 0) ? 1u : 0u);
    };
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_full(0), 0, 4, abort_flag));
      if (ok) {
        tc_fence_after();
        issue_sdp(0, 0);
        issue_sdp(0, 1);
      }
    }
    for (int u = 0; ok && u < n; ++u) {
      const int s = u % C::kStages, s1 = (u + 1) % C::kStages;
      const bool more = u + 1 < n;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_pp0, u & 1, 5, abort_flag)))) break;
      tc_fence_after();
      issue_acc(s, 0, u == 0);
      if (more) {
        if (!(ok = __all_sync(0xffffffffu,
                              mbar_wait(bar_full(s1), ((u + 1) / C::kStages) & 1, 4, abort_flag))))
          break;
        tc_fence_after();
        issue_sdp(s1, 0);
      }
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_pp0 + 8, u & 1, 5, abort_flag)))) break;
      tc_fence_after();
      issue_acc(s, 1, false);
      umma_commit_elect(bar_empty(s));
      if (more) issue_sdp(s1, 1);
      else umma_commit_elect(bar_acc);
    }
    umma_commit_elect(bar_drain);
    mbar_wait(bar_drain, 0, 6);
    __syncwarp();
  } else {
    // --------------------------------------------------------- elementwise
    const int r = threadIdx.x;  // key row within the tile = TMEM lane
    const int kj = k0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float* st_lse = stats + warp * 2 * kBM;  // this warp's copy of the tile statistics
    float* st_dlt = st_lse + kBM;
    const float sl2 = p.scale_log2;
    const float2 sl2x2 = make_float2(sl2, sl2);
    const bool key_ok = kj < L;
    const bool keys_ok = __all_sync(0xffffffffu, key_ok);
    const int kj_warp_max = k0 + warp * 32 + 31;
    // LSE*log2e and delta of item u's 128 query rows, 4 per lane; rows that
    // are past T or padded get lse = +inf (P = 0).  Loaded one item ahead.
    float nl[4], nd[4];
    auto fetch = [&](int u) {
      const int hq = g * G + u / n_tiles_per_head;
      const int q0 = (i_lo + u % n_tiles_per_head) * kBM;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = q0 + lane + 32 * e;
        const bool valid = i < p.T && i + off < L;
        const size_t row = ((size_t)b * p.Hq + hq) * p.T + i;
        nl[e] = valid ? p.lse[row] * 1.4426950408889634f : INFINITY;
        nd[e] = valid ? p.delta[row] : 0.f;
      }
    };
    if (n > 0) fetch(0);
    bool ok = true;
    for (int u = 0; ok && u < n; ++u) {
      const int q0 = (i_lo + u % n_tiles_per_head) * kBM;
      __syncwarp();
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        st_lse[lane + 32 * e] = nl[e];
        st_dlt[lane + 32 * e] = nd[e];
      }
      __syncwarp();
      if (u + 1 < n) fetch(u + 1);
      // key kj is visible to query column c iff kj < L and (not causal or
      // kj <= q0 + c + off); invalid columns already have lse = +inf.
      const int c_min = p.causal ? kj - q0 - off : -1;  // visible columns: c >= c_min
      const int c_min_warp = p.causal ? kj_warp_max - q0 - off : -1;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar_mm0 + 8u * hh, u & 1, 7, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const int cb = hh * kHalf;  // first query column of the half
        // every (key, query) pair of the half visible for the whole warp
        const int last = q0 + cb + kHalf - 1;
        const bool dense = keys_ok && c_min_warp <= cb && last < p.T && last + off < L;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t sr[32], dp[32];
          tmem_ld32(lane_base + col_s(hh) + 32 * c, sr);
          tmem_ld32(lane_base + col_dp(hh) + 32 * c, dp);
          tmem_wait_ld32(sr);
          tmem_wait_ld32(dp);
          uint32_t ppk[16], dpk[16];
          const float* sl = st_lse + cb + 32 * c;
          const float* sd = st_dlt + cb + 32 * c;
          if (dense) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 l = *reinterpret_cast<const float2*>(sl + e);
              const float2 dl = *reinterpret_cast<const float2*>(sd + e);
              const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                          sl2x2, make_float2(-l.x, -l.y));
              const float2 pe = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              const float2 d = __fadd2_rn(make_float2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])),
                                          make_float2(-dl.x, -dl.y));
              const float2 ds = __fmul2_rn(pe, d);
              ppk[e >> 1] = pack2<kF16>(pe.x, pe.y);
              dpk[e >> 1] = pack2<kF16>(ds.x, ds.y);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const int col = cb + 32 * c + e;
              const float l0 = sl[e], l1 = sl[e + 1];
              // selects, not products: hidden entries may hold NaN
              const bool v0 = key_ok && col >= c_min && l0 != INFINITY;
              const bool v1 = key_ok && col + 1 >= c_min && l1 != INFINITY;
              const float e0 = ex2_approx(fmaf(__uint_as_float(sr[e]), sl2, -l0));
              const float e1 = ex2_approx(fmaf(__uint_as_float(sr[e + 1]), sl2, -l1));
              const float p0 = v0 ? e0 : 0.f, p1 = v1 ? e1 : 0.f;
              const float d0 = v0 ? e0 * (__uint_as_float(dp[e]) - sd[e]) : 0.f;
              const float d1 = v1 ? e1 * (__uint_as_float(dp[e + 1]) - sd[e + 1]) : 0.f;
              ppk[e >> 1] = pack2<kF16>(p0, p1);
              dpk[e >> 1] = pack2<kF16>(d0, d1);
            }
          }
          tmem_st16(lane_base + col_s(hh) + 16 * c, ppk);
          tmem_st16(lane_base + col_dp(hh) + 16 * c, dpk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_pp0 + 8u * hh);
      }
    }
    // ------------------------------------------------------------ epilogue
    if (ok && n > 0) ok = __all_sync(0xffffffffu, mbar_wait(bar_acc, 0, 8, abort_flag));
    const bool has = ok && n > 0;
    if (has) tc_fence_after();
    const size_t krow = ((size_t)b * p.Hkv + g) * p.S + kj;
#pragma unroll
    for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK
      uint16_t* drow = reinterpret_cast<uint16_t*>(which ? p.dk : p.dv) + krow * D;
      const float sc = which ? p.scale : 1.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t a[32];
        if (has) {
          tmem_ld32(lane_base + (which ? kColDK : kColDV) + 32 * c, a);
          tmem_wait_ld32(a);
        }
        if (kj < p.S) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 w = make_uint4(0, 0, 0, 0);
            if (has) {
              w.x = pack2<kF16>(__uint_as_float(a[8 * v4 + 0]) * sc, __uint_as_float(a[8 * v4 + 1]) * sc);
              w.y = pack2<kF16>(__uint_as_float(a[8 * v4 + 2]) * sc, __uint_as_float(a[8 * v4 + 3]) * sc);
              w.z = pack2<kF16>(__uint_as_float(a[8 * v4 + 4]) * sc, __uint_as_float(a[8 * v4 + 5]) * sc);
              w.w = pack2<kF16>(__uint_as_float(a[8 * v4 + 6]) * sc, __uint_as_float(a[8 * v4 + 7]) * sc);
            }
            reinterpret_cast<uint4*>(drow + 32 * c)[v4] = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace tcbwd
}  // namespace attn
