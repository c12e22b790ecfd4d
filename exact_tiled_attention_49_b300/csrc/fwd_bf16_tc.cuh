// fwd_bf16_tc.cuh -- bf16 prefill forward on the 5th-generation tensor cores.
//
// The method ("FlashAttention", Transformers in Action section 9.4.1 and
// Figure 9.8; "Implementing attention from scratch", Core ideas, Stable
// softmax): a tile of BM query rows stays on chip while BN-key tiles of K and
// V stream past it; per row a running maximum m and denominator l are kept
// and the partial output is rescaled by exp(m_old - m_new) when m grows, so
// the T x S score matrix never reaches HBM.
//
// Mapping to sm_103a, one CTA per (query tile, head, batch):
//   warp 4      TMA producer: Q once, then K_0, K_1, V_0, K_2, V_1, ... into a
//               ring of NSLOT shared-memory slots (128B-swizzled tiles).
//   warp 5      MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//               score buffers (tcgen05.mma, bf16 in, fp32 accumulate), and
//               O += P_j V_j with P_j read from TMEM as the A operand.
//   warps 0-3   softmax: thread r owns TMEM lane r = query row r.  It loads
//               its 128 scores, applies the causal/padding mask on boundary
//               tiles only, updates m and l, writes P_j = exp2(x - m) as bf16
//               over the first 64 columns of the score buffer, and rescales
//               the O row in TMEM when needed.  Epilogue: O / l and the LSE.
// TMEM (512 columns): S buffers at columns 0 and 128, O at column 256.
//
// Rescaling is lazy: the exponent reference m_ref moves only when a row's
// maximum exceeds it by more than kRescaleThreshold (log2 units), so P can
// reach 2^8 but O, l and m_ref always stay consistent and the final O / l is
// exact up to rounding.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace attn {
namespace tcfwd {

constexpr int kBM = 128;              // query rows per CTA (= TMEM lanes)
constexpr int kBN = 128;              // keys per tile
constexpr int kThreads = 192;         // 4 softmax warps + load warp + MMA warp
constexpr int kLoadWarp = 4;
constexpr int kMmaWarp = 5;
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;                    // 64-column (128 B) chunks
  static constexpr uint32_t kTileBytes = kBN * D * 2;       // one K or V tile
  static constexpr uint32_t kChunkBytes = kBN * 128;        // 128 rows x 128 B
  static constexpr uint32_t kQBytes = kBM * D * 2;
  static constexpr int kSlots = (D == 128) ? 5 : 8;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffSlots = kQBytes;
  static constexpr uint32_t kOffBars = kOffSlots + kSlots * kTileBytes;
  // barriers: q_full, slot_full[S], slot_empty[S], s_full[2], p_full, o_done, drain
  static constexpr int kNumBars = 1 + 2 * kSlots + 2 + 3;
  static constexpr uint32_t kOffMisc = kOffBars + 8 * kNumBars;
  static constexpr uint32_t kBytes = kOffMisc + 16;
  static constexpr size_t kSmemAlloc = kBytes + 1024;       // + alignment slack
};

struct Params {
  void* o;                  // [B,Hq,T,D] bf16
  float* lse;               // [B,Hq,T] or null
  const int32_t* key_lens;  // [B] or null
  int B, Hq, Hkv, T, S;
  int causal;
  int n_qtiles;
  float scale_log2;         // scale * log2(e)
};

// Number of key tiles the query tile starting at q0 must visit, and its valid
// key bound L.  Shared by all roles so they agree on the trip count.
__device__ __forceinline__ int tile_count(const Params& p, int b, int q0, int& L) {
  L = p.S;
  if (p.key_lens != nullptr) L = min(max(p.key_lens[b], 0), p.S);
  const int off = p.S - p.T;
  if (q0 + off >= L) return 0;  // every row of the tile is a padded row
  int kv_end = L;
  if (p.causal) kv_end = min(L, q0 + kBM + off);  // last row sees keys <= q0+BM-1+off
  if (kv_end <= 0) return 0;
  return (kv_end + kBN - 1) / kBN;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t s_q = sbase + C::kOffQ;
  const uint32_t s_slots = sbase + C::kOffSlots;
  const uint32_t bars = sbase + C::kOffBars;
  const uint32_t bar_q = bars;
  auto bar_full = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_empty = [&](int s) { return bars + 8u * (1 + C::kSlots + s); };
  const uint32_t bar_s0 = bars + 8u * (1 + 2 * C::kSlots);
  const uint32_t bar_p = bar_s0 + 16;
  const uint32_t bar_o = bar_p + 8;
  const uint32_t bar_drain = bar_o + 8;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = p.n_qtiles - 1 - (int)blockIdx.x;  // heaviest causal tiles first
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (p.Hq / p.Hkv);
  const int q0 = qt * kBM;
  int L;
  const int n = tile_count(p, b, q0, L);
  const int off = p.S - p.T;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_s0, 1);
    mbar_init(bar_s0 + 8, 1);
    mbar_init(bar_p, 4 * 32);
    mbar_init(bar_o, 1);
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

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      const int bh_q = b * p.Hq + h;
      const int bh_kv = b * p.Hkv + g;
      mbar_arrive_expect_tx(bar_q, C::kQBytes);
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_3d(s_q + c * C::kChunkBytes, &tm_q, bar_q, c * 64, q0, bh_q);
      // Load order = consumption order: K_0, then (K_j, V_{j-1}) for j >= 1,
      // then V_{n-1}.
      const int total = 2 * n;
      int last_issue[C::kSlots];
      for (int s = 0; s < C::kSlots; ++s) last_issue[s] = -1;
      for (int t = 0; t < total; ++t) {
        bool is_v;
        int tile;
        if (t == 0) { is_v = false; tile = 0; }
        else if (t == total - 1) { is_v = true; tile = n - 1; }
        else if (t & 1) { is_v = false; tile = (t + 1) >> 1; }
        else { is_v = true; tile = (t >> 1) - 1; }
        const int slot = t % C::kSlots;
        if (t >= C::kSlots) {
          if (!mbar_wait(bar_empty(slot), ((t / C::kSlots) - 1) & 1, 1, abort_flag)) break;
        }
        const uint32_t dst = s_slots + slot * C::kTileBytes;
        mbar_arrive_expect_tx(bar_full(slot), C::kTileBytes);
        const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(dst + c * C::kChunkBytes, tm, bar_full(slot), c * 64, tile * kBN, bh_kv);
        last_issue[slot] = t;
      }
      // Drain: every issued copy must land before the CTA may exit.
      for (int s = 0; s < C::kSlots; ++s)
        if (last_issue[s] >= 0) mbar_wait(bar_full(s), (last_issue[s] / C::kSlots) & 1, 2);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(kBM, D, false, true);
      bool ok = mbar_wait(bar_q, 0, 3, abort_flag);
      int t = 0;  // consumption counter (same order as the loads)
      auto wait_slot = [&](int tt) {
        return mbar_wait(bar_full(tt % C::kSlots), (tt / C::kSlots) & 1, 4, abort_flag);
      };
      auto issue_qk = [&](int tt, int buf) {
        const uint32_t kt = s_slots + (tt % C::kSlots) * C::kTileBytes;
        const uint32_t d_tmem = tmem + (buf ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          umma_ss(d_tmem, sdesc_sw128(s_q + koff, 16, 1024), sdesc_sw128(kt + koff, 16, 1024),
                  idesc_qk, kk > 0);
        }
        umma_commit(bar_s0 + 8 * buf);
        umma_commit(bar_empty(tt % C::kSlots));
      };
      if (ok && (ok = wait_slot(t))) {
        tc_fence_after();
        issue_qk(t, 0);
        ++t;
      }
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) {
          if (!(ok = wait_slot(t))) break;
          tc_fence_after();
          issue_qk(t, (j + 1) & 1);
          ++t;
        }
        if (!(ok = mbar_wait(bar_p, j & 1, 5, abort_flag))) break;
        if (!(ok = wait_slot(t))) break;
        tc_fence_after();
        const uint32_t vt = s_slots + (t % C::kSlots) * C::kTileBytes;
        const uint32_t p_tmem = tmem + ((j & 1) ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          umma_ts(tmem + kColO, p_tmem + kk * 8, sdesc_sw128(vt + kk * 2048, C::kChunkBytes, 1024),
                  idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar_o);
        umma_commit(bar_empty(t % C::kSlots));
        ++t;
      }
      // Drain: all issued MMAs complete before TMEM is released.
      umma_commit(bar_drain);
      mbar_wait(bar_drain, 0, 6);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int r = threadIdx.x;  // query row within the tile = TMEM lane
    const int i = q0 + r;
    const int pos = i + off;
    const bool row_ok = (i < p.T) && (pos < L);
    const int lim = p.causal ? min(L, pos + 1) : L;  // visible keys: [0, lim)
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY;  // exponent reference (log2 units)
    float l = 0.f;
    bool ok = true;

    for (int j = 0; j < n; ++j) {
      const int buf = j & 1;
      ok = mbar_wait(bar_s0 + 8 * buf, (j >> 1) & 1, 7, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t ts = lane_base + (buf ? kColS1 : kColS0);
      uint32_t sr[kBN];
      tmem_ld32(ts + 0, sr + 0);
      tmem_ld32(ts + 32, sr + 32);
      tmem_ld32(ts + 64, sr + 64);
      tmem_ld32(ts + 96, sr + 96);
      tmem_wait_ld32(sr + 0);
      tmem_wait_ld32(sr + 32);
      tmem_wait_ld32(sr + 64);
      tmem_wait_ld32(sr + 96);

      const int k0 = j * kBN;
      const bool masked = (k0 + kBN > L) || (p.causal && (k0 + kBN - 1 > q0 + off));
      float mx = -INFINITY;
      if (masked) {
#pragma unroll
        for (int c = 0; c < kBN; ++c) {
          if (k0 + c >= lim) sr[c] = __float_as_uint(-INFINITY);
          mx = fmaxf(mx, __uint_as_float(sr[c]));
        }
      } else {
#pragma unroll
        for (int c = 0; c < kBN; ++c) mx = fmaxf(mx, __uint_as_float(sr[c]));
      }
      const float m_tile = mx * sl2;  // -inf stays -inf (sl2 > 0)

      // Lazy rescale: move the reference only when the maximum ran ahead.
      const bool first = (m_ref == -INFINITY);
      const bool grow = !first && (m_tile > m_ref + kRescaleThreshold);
      if (first && m_tile != -INFINITY) m_ref = m_tile;
      if (__any_sync(0xffffffffu, grow)) {
        // O holds P_{j-1} V_{j-1} only once that MMA has completed.
        ok = mbar_wait(bar_o, (j - 1) & 1, 8, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float alpha = grow ? ex2_approx(m_ref - m_tile) : 1.f;
        if (grow) {
          l *= alpha;
          m_ref = m_tile;
        }
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(lane_base + kColO + 32 * c, orr);
          tmem_wait_ld32(orr);
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
          tmem_st32(lane_base + kColO + 32 * c, orr);
        }
      }

      const float neg_ref = (m_ref == -INFINITY) ? 0.f : -m_ref;
      float sum = 0.f;
      uint32_t pk[kBN / 2];
#pragma unroll
      for (int c = 0; c < kBN; c += 2) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c]), sl2, neg_ref));
        const float p1 = ex2_approx(fmaf(__uint_as_float(sr[c + 1]), sl2, neg_ref));
        sum += p0 + p1;
        pk[c >> 1] = pack_bf16x2(p0, p1);
      }
      l += sum;
      tmem_st32(ts + 0, pk);
      tmem_st32(ts + 32, pk + 32);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_p);
    }

    // ------------------------------------------------------------ epilogue
    if (ok && n > 0) {
      ok = mbar_wait(bar_o, (n - 1) & 1, 9, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
    }
    const bool has = ok && row_ok && (l > 0.f);
    const float inv = has ? 1.f / l : 0.f;
    __nv_bfloat16* orow =
        reinterpret_cast<__nv_bfloat16*>(p.o) + ((((size_t)b * p.Hq + h) * p.T) + i) * D;
    if (__any_sync(0xffffffffu, has)) {
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t orr[32];
        tmem_ld32(lane_base + kColO + 32 * c, orr);
        tmem_wait_ld32(orr);
        if (!has) {
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = 0u;
        }
        if (i < p.T) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 u;
            u.x = pack_bf16x2(__uint_as_float(orr[8 * v + 0]) * inv, __uint_as_float(orr[8 * v + 1]) * inv);
            u.y = pack_bf16x2(__uint_as_float(orr[8 * v + 2]) * inv, __uint_as_float(orr[8 * v + 3]) * inv);
            u.z = pack_bf16x2(__uint_as_float(orr[8 * v + 4]) * inv, __uint_as_float(orr[8 * v + 5]) * inv);
            u.w = pack_bf16x2(__uint_as_float(orr[8 * v + 6]) * inv, __uint_as_float(orr[8 * v + 7]) * inv);
            dst[v] = u;
          }
        }
      }
    } else if (i < p.T) {
      uint4* dst = reinterpret_cast<uint4*>(orow);
      for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0, 0, 0, 0);
    }
    if (p.lse != nullptr && i < p.T) {
      p.lse[((size_t)b * p.Hq + h) * p.T + i] =
          has ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace tcfwd
}  // namespace attn
