// fwd_bf16_tc.cuh -- bf16 / fp16 / E4M3 prefill forward on the 5th-generation
// tensor cores.
//
// The method ("FlashAttention", Transformers in Action section 9.4.1 and
// Figure 9.8; "Implementing attention from scratch", Core ideas, Stable
// softmax): a tile of query rows stays on chip while 128-key tiles of K and V
// stream past it; per row a running maximum m and denominator l are kept and
// the partial output is rescaled by exp(m_old - m_new) when m grows, so the
// T x S score matrix never reaches HBM.
//
// Mapping to sm_103a.  The kernel is persistent, one CTA per SM; an item is a
// pair of 128-row query tiles (rows q0 .. q0 + 255) of one (batch, head),
// paired from the top of the sequence's non-padded rows (so q0 may be -128:
// a virtual first tile), and the items, numbered heaviest first, are dealt
// to the CTAs in snake order so that causal work balances over the SMs
// (sched_next).  Per CTA:
//   warps 0-3   softmax of query tile 0, warps 4-7 softmax of query tile 1:
//               thread r of a group owns TMEM lane r = query row r of its
//               tile.  It loads its 128 scores, masks diagonal/boundary tiles
//               only, updates m and l, writes P = exp2(x - m) as bf16 over
//               the first 64 columns of its score buffer, rescales its O row
//               in TMEM when needed, and at the end of the item writes O / l
//               and the LSE.
//   warp 8      MMA issuer (one thread): S_t = Q_t K_j^T into TMEM score
//               buffer t (tcgen05.mma, bf16 in, fp32 accumulate) and
//               O_t += P_t V_j with P_t read from TMEM as the A operand.
//   warp 9      TMA producer: Q_0, Q_1 once per item, then K_0, V_0, K_1,
//               V_1, ... into a ring of 128B-swizzled shared-memory slots.
//               With a causal diagonal (tile 1 visits one key tile more) the
//               next item's Q_0 and K_0 go out between this item's last K
//               and last V, and the MMA warp starts the next item's S_0
//               while tile 1 finishes alone.
// The two query tiles share every K/V tile and take turns on the tensor
// cores: while group 0 turns S_0 into P_0, the tensor cores compute P_1 V and
// the next S_1, and the other way round.  Issue order per key tile j:
//   PV_0(j), S_0(j+1), PV_1(j), S_1(j+1).
// tcgen05 operations issued by one thread run in order, so when S_t(j+1) has
// completed, PV_t(j) has too: the softmax group may rescale O_t right after
// its score wait, and S_t(j+1) may overwrite the P_t(j) that PV_t(j) read.
// TMEM (512 columns): S_0 at 0, S_1 at 128, O_0 at 256, O_1 at 256 + D.
//
// Rescaling is lazy: the exponent reference m_ref moves only when a row's
// maximum exceeds it by more than kRescaleThreshold (log2 units), so P can
// reach 2^8 but O, l and m_ref always stay consistent and the final O / l is
// exact up to rounding.  E4M3 inputs use kind::f8f6f4 MMAs and round P to
// E4M3 (see the kF8 notes at the kernel).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace attn {
namespace tcfwd {

constexpr int kBM = 128;              // query rows per tile (= TMEM lanes)
constexpr int kQTiles = 2;            // query tiles per work item
constexpr int kItemRows = kBM * kQTiles;
constexpr int kBN = 128;              // keys per tile
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kThreads = 320;         // 8 softmax warps + MMA warp + load warp
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kTmemCols = 512;

// EB: bytes per input element (2: bf16 / fp16, 1: E4M3).
template <int D, int EB = 2>
struct Cfg {
  static constexpr int kRowBytes = D * EB;                  // one Q, K or V row
  static constexpr int kChunks = kRowBytes / 128;           // 128-byte swizzle chunks per row
  static constexpr int kChunkElems = 128 / EB;              // elements of a chunk row
  static constexpr uint32_t kTileBytes = kBN * kRowBytes;   // one K or V tile
  static constexpr uint32_t kChunkBytes = kBN * 128;        // 128 rows x 128 B
  static constexpr uint32_t kQBytes = kBM * kRowBytes;      // one query tile
  static constexpr int kKSteps = kRowBytes / 32;            // S = Q K^T: 32-byte K steps
  static constexpr int kPvSteps = kBN * EB / 64;            // P V per 64-key half: 32-byte steps
  static constexpr int kSlots = (kTileBytes >= 32768) ? 5 : 8;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffSlots = kQTiles * kQBytes;
  static constexpr uint32_t kOffBars = kOffSlots + kSlots * kTileBytes;
  // barriers: q_full[2], q_empty[2], slot_full[S], slot_empty[S], s_full[2],
  // p_half[2][2], o_full[2], drain, tail
  static constexpr int kNumBars = 2 + 2 + 2 * kSlots + 2 + 4 + 2 + 1 + 1;
  static constexpr uint32_t kOffMisc = kOffBars + 8 * kNumBars;    // TMEM address, abort flag
  static constexpr uint32_t kOffSched = (kOffMisc + 16 + 15) / 16 * 16;  // SchedArgs
  static constexpr uint32_t kOffWalk = kOffSched + 64;                   // WalkState[warps][2]
  static constexpr uint32_t kBytes = kOffWalk + 32 * 2 * (kThreads / 32);
  static constexpr size_t kSmemAlloc = kBytes + 1024;       // + alignment slack
  static constexpr uint32_t kColS(int t) { return (uint32_t)(t * kBN); }
  static constexpr uint32_t kColO(int t) { return (uint32_t)(2 * kBN + t * D); }
};

struct Params {
  void* o;                  // [B,Hq,T,D] bf16 or fp16
  float* lse;               // [B,Hq,T] or null
  const int32_t* key_lens;  // [B] or null
  const int32_t* q_pos;     // [B] key position of query row 0, or null (S - T)
  int B, Hq, Hkv, T, S;
  int causal;
  int k_off;                // global position of key row 0 (sharded keys; else 0)
  int shard;                // key_lens / q_pos are global positions (see seq_geom)
  int n_pairs;              // pair slots per (batch, head): enough for T + 128 rows
                            // when a sequence's pairs may be shifted
  int n_items;              // n_pairs * B * Hq
  int o_align32;            // o is 32-byte aligned: 256-bit stores
  float scale_log2;         // scale * log2(e) (E4M3: times the Q and K descales)
  float o_scale;            // factor on O (E4M3: the V descale; else 1)
  FastDiv div_B, div_Hq, div_G;  // division by B, Hq and Hq / Hkv
};

struct Item {
  int b, h, q0;             // q0 = first row of query tile 0
};

// Geometry of sequence b (common.cuh, seq_geom): valid key bound L, query
// offset off (row i sits at key i + off) and non-padded row count R.
__device__ __forceinline__ SeqGeom geom(const Params& p, int b) {
  return seq_geom(p.key_lens, p.q_pos, p.k_off, p.shard != 0, b, p.T, p.S);
}

// Pairing of query tiles.  The query tiles of a sequence that hold at least
// one non-padded row are paired from the top: when their count is odd, every
// pair of the sequence starts 128 rows lower (the shift), so the tile left
// without a partner is tile 0, which visits the fewest key tiles under a
// causal mask, instead of the last and heaviest one.  A shifted sequence's
// first pair then has a virtual tile at rows -128..-1, which has no rows, no
// key tiles and no loads.
__device__ __forceinline__ int seq_shift(int T, int R) {
  const int rows = min(T, R);  // rows below this are not padded
  const int tiles = rows > 0 ? (rows + kBM - 1) / kBM : 0;
  return (tiles & 1) ? kBM : 0;
}

// Number of key tiles the query tile starting at row q0 must visit (0 when
// every row of the tile is past T, padded, virtual or sees no key), for the
// sequence geometry g.  Every role computes it the same way so they agree on
// the trip counts.
__device__ __forceinline__ int tile_count(const Params& p, int q0, const SeqGeom& g) {
  if (q0 < 0 || q0 >= p.T) return 0;
  if (q0 >= g.R) return 0;  // every row of the tile is a padded row
  int kv_end = g.L;
  if (p.causal) kv_end = min(g.L, q0 + kBM + g.off);  // last row sees keys <= q0+BM-1+off
  if (kv_end <= 0) return 0;
  return (kv_end + kBN - 1) / kBN;
}

// Sizes the work walk needs, copied once into shared memory, and one walk
// state per warp.  The walk is a non-inlined function that takes only
// shared-memory pointers: passing the kernel parameters by reference to a
// non-inlined function would move them to local memory, and every later
// parameter read in the kernel would become a slow local load.
struct SchedArgs {
  const int32_t* key_lens;
  const int32_t* q_pos;
  int n_pairs, B, Hq, T, S;
  int flags;      // kCausal | kAllBusy | kShard
  FastDiv div_B, div_Hq;
  int shift_all;  // the shift of every sequence (closed-form walk)
  int k_off;
};
enum : int { kCausal = 1, kAllBusy = 2, kShard = 4 };
static_assert(sizeof(SchedArgs) <= 64, "SchedArgs fits its shared-memory slot");
struct WalkState {
  int g0;         // first group of the current 32-group window
  int base;       // list index of the window's first item
  int round;      // items handed out so far
  int have;       // `mask` holds the current window's classification
  uint32_t mask;  // groups of the window that are in the list (bit = lane)
  uint32_t smask; // groups of the window whose sequence is shifted
  int pad[2];
};

// Key tiles of the query tile starting at q0 (the rule of tile_count).
__device__ __forceinline__ int sched_tiles(const SchedArgs& a, int q0, const SeqGeom& g) {
  if (q0 < 0 || q0 >= a.T || q0 >= g.R) return 0;
  const int kv_end = (a.flags & kCausal) ? min(g.L, q0 + kBM + g.off) : g.L;
  return kv_end <= 0 ? 0 : (kv_end + kBN - 1) / kBN;
}

// Next work item of this CTA, packed as valid << 63 | shifted << 62 |
// pair << 32 | b << 16 | h (0 when there is none).
//
// The items are ordered pair-descending (the heaviest causal work first),
// then by batch and head; a "group" is the Hq items of one (pair, batch).
// Items with at least one key tile to visit are dealt out in snake order over
// the compacted list of such items: CTA c of G takes positions c, 2G-1-c,
// 2G+c, 4G-1-c, ...  With causal masking and key padding this list is
// sorted by cost, so the snake keeps the per-SM sums of work within a few
// percent of each other.  Items with nothing to visit (every row padded or
// past T) form a second list (kEmpty), dealt out round-robin (c, c+G, ...);
// their rows are only zeroed.
//
// Called by a whole converged warp; every lane gets the same item.  Without
// key padding and with T <= S (or no causal mask) no group is empty and the
// item follows from its position in closed form; otherwise the warp
// classifies 32 groups per step (ballot + prefix count), because a serial
// walk costs about 200 cycles per group.  The classification of the current
// window is kept in the walk state, and the divisions by B and Hq are
// multiply-highs: a walk that reclassified its window and divided with the
// divide sequence on every call took 2000-3700 cycles of the MMA warp at each
// item boundary, mostly waiting behind the softmax warps' exponentials.
// Every role of the CTA walks its own copy and sees the same sequence.
template <bool kEmpty>
__device__ __noinline__ uint64_t sched_next(const SchedArgs* args, WalkState* st) {
  const SchedArgs a = *args;
  const int G = gridDim.x, c = blockIdx.x;
  const int round = st->round;
  const int target = kEmpty ? round * G + c : round * G + ((round & 1) ? (G - 1 - c) : c);
  const int n_groups = a.n_pairs * a.B;
  const int lane = threadIdx.x & 31;
  __syncwarp();
  if (lane == 0) st->round = round + 1;
  if (a.flags & kAllBusy) {
    __syncwarp();
    if (kEmpty || target >= n_groups * a.Hq) return 0;
    const int g = fast_div(target, a.div_Hq);
    const int pr = fast_div(g, a.div_B);
    return (1ull << 63) | ((uint64_t)(a.shift_all != 0) << 62) |
           ((uint64_t)(a.n_pairs - 1 - pr) << 32) | ((uint64_t)(g - pr * a.B) << 16) |
           (uint64_t)(target - g * a.Hq);
  }
  int g0 = st->g0, base = st->base, have = st->have;
  uint32_t mask = st->mask, smask = st->smask;
  uint64_t res = 0;
  while (g0 < n_groups) {
    if (!have) {
      const int g = g0 + lane;
      bool in_list = false, shifted = false;
      if (g < n_groups) {
        const int pr = fast_div(g, a.div_B), b = g - pr * a.B;
        const SeqGeom sg = seq_geom(a.key_lens, a.q_pos, a.k_off, (a.flags & kShard) != 0, b,
                                    a.T, a.S);
        const int sh = seq_shift(a.T, sg.R);
        const int q0 = (a.n_pairs - 1 - pr) * kItemRows - sh;
        const bool busy = sched_tiles(a, q0, sg) > 0 || sched_tiles(a, q0 + kBM, sg) > 0;
        in_list = busy != kEmpty;
        shifted = sh != 0;
      }
      mask = __ballot_sync(0xffffffffu, in_list);
      smask = __ballot_sync(0xffffffffu, shifted);
      have = 1;
    }
    const int cnt = __popc(mask) * a.Hq;
    if (target < base + cnt) {
      // the k-th set bit of the mask is the group that holds the target
      const int k = fast_div(target - base, a.div_Hq);
      const bool mine = ((mask >> lane) & 1u) && __popc(mask & ((1u << lane) - 1u)) == k;
      const int ls = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
      const int gs = g0 + ls;
      const int pr = fast_div(gs, a.div_B);
      res = (1ull << 63) | ((uint64_t)((smask >> ls) & 1u) << 62) |
            ((uint64_t)(a.n_pairs - 1 - pr) << 32) | ((uint64_t)(gs - pr * a.B) << 16) |
            (uint64_t)(target - base - k * a.Hq);
      break;  // later targets are larger: keep this window
    }
    base += cnt;
    g0 += 32;
    have = 0;
  }
  if (lane == 0) {
    st->g0 = g0;
    st->base = base;
    st->have = have;
    st->mask = mask;
    st->smask = smask;
  }
  __syncwarp();
  return res;
}

// Unpacks a sched_next result; false when the walk is over.
__device__ __forceinline__ bool unpack_item(uint64_t v, Item& it) {
  if (!(v >> 63)) return false;
  it.q0 = (int)((v >> 32) & 0x3FFFFFFFu) * kItemRows - (int)((v >> 62) & 1u) * kBM;
  it.b = (int)((v >> 16) & 0xFFFFu);
  it.h = (int)(v & 0xFFFFu);
  return true;
}

// Zero rows [r0, kBN) of a K/V slot at shared address `slot` (kChunks
// 128-byte column chunks of kBN rows each; a whole 128-byte row is zeroed,
// so the swizzle does not matter), then make the writes visible to the
// tensor cores.  Whole warp.
template <int kChunks>
__device__ __forceinline__ void zero_rows_from(uint32_t slot, int r0, int lane) {
  for (int idx = r0 * 8 + lane; idx < kBN * 8; idx += 32)
#pragma unroll
    for (int c = 0; c < kChunks; ++c) st_shared_zero16(slot + c * (kBN * 128) + idx * 16);
  fence_proxy_async_shared();
  __syncwarp();
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// kF16: fp16 inputs and output (else bf16); both use kind::f16 MMAs.
// kF8: E4M3 inputs (kind::f8f6f4 MMAs, P rounded to E4M3 for P V), bf16
// output.  P is formed against a reference 7 below the row maximum's
// (P' = 2^7 P), so the weights that matter stay in E4M3's normal range (down
// to 2^-13 of the largest); with the lazy-rescale threshold at 1 the largest
// P' is 2^8 < 448.  O / l and the LSE use the same biased reference, so the
// bias cancels exactly.
template <int D, bool kF16, bool kF8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, Params p) {
  static_assert(!(kF16 && kF8), "E4M3 inputs write bf16 output");
  using C = Cfg<D, kF8 ? 1 : 2>;
  constexpr float kPBias = kF8 ? 7.f : 0.f;                      // log2 of P's scale
  constexpr float kThresh = kF8 ? 1.f : kRescaleThreshold;       // lazy-rescale threshold
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t s_q = sbase + C::kOffQ;
  const uint32_t s_slots = sbase + C::kOffSlots;
  const uint32_t bars = sbase + C::kOffBars;
  auto bar_qfull = [&](int t) { return bars + 8u * t; };
  auto bar_qempty = [&](int t) { return bars + 8u * (2 + t); };
  auto bar_full = [&](int s) { return bars + 8u * (4 + s); };
  auto bar_empty = [&](int s) { return bars + 8u * (4 + C::kSlots + s); };
  const uint32_t bar_s = bars + 8u * (4 + 2 * C::kSlots);  // s_full[t] = bar_s + 8t
  const uint32_t bar_p = bar_s + 16;                        // p_half[t][h] = bar_p + 16t + 8h
  const uint32_t bar_o = bar_p + 32;                        // o_full[t]
  const uint32_t bar_drain = bar_o + 16;
  const uint32_t bar_tail = bar_drain + 8;  // producer-private: the V tile that straddles L
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  SchedArgs* sched = reinterpret_cast<SchedArgs*>(smem + C::kOffSched);
  // walk[0]: this warp's list of work items, walk[1]: its list of empty items
  WalkState* walk = reinterpret_cast<WalkState*>(smem + C::kOffWalk) + 2 * (threadIdx.x >> 5);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(bar_qfull(t), 1);
      mbar_init(bar_qempty(t), 1);
      mbar_init(bar_s + 8 * t, 1);
      mbar_init(bar_p + 16 * t, 4 * 32);
      mbar_init(bar_p + 16 * t + 8, 4 * 32);
      mbar_init(bar_o + 8 * t, 1);
    }
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_tail, 1);
    *abort_flag = 0;
    fence_mbar_init();
    sched->key_lens = p.key_lens;
    sched->q_pos = p.q_pos;
    sched->n_pairs = p.n_pairs;
    sched->B = p.B;
    sched->Hq = p.Hq;
    sched->T = p.T;
    sched->S = p.S;
    sched->div_B = p.div_B;
    sched->div_Hq = p.div_Hq;
    sched->shift_all = seq_shift(p.T, p.T);
    sched->k_off = p.k_off;
    const bool all_busy =
        p.key_lens == nullptr && p.q_pos == nullptr && (!p.causal || p.T <= p.S);
    sched->flags = (p.causal ? kCausal : 0) | (all_busy ? kAllBusy : 0) | (p.shard ? kShard : 0);
  }
  if (lane == 0) walk[0] = walk[1] = WalkState{0, 0, 0, 0, 0u, 0u, {0, 0}};
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
    // The whole warp walks the schedule and waits; lane 0 issues the copies.
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
    }
    int ring = 0, qi = 0, ntail = 0;
    int nq0 = 0, nq1 = 0;  // phases armed so far on q_full[0] and q_full[1]
    bool ok = true;
    auto wait_bar = [&](uint32_t bar, uint32_t parity) {
      const bool w = mbar_wait(bar, parity, 1, abort_flag);
      return __all_sync(0xffffffffu, w);
    };
    // Next item with key tiles to visit (false when the walk is over).
    auto next_item = [&](Item& x, int& L, int& n0, int& n1) {
      while (unpack_item(sched_next<false>(sched, walk), x)) {
        const SeqGeom g = geom(p, x.b);
        L = g.L;
        n0 = tile_count(p, x.q0, g);
        n1 = tile_count(p, x.q0 + kBM, g);
        if (max(n0, n1) > 0) return true;
      }
      return false;
    };
    // Query tile t of the item with row x.q0 into its buffer (qi-th use).
    auto load_q = [&](const Item& x, int t) {
      if (qi > 0 && !(ok = wait_bar(bar_qempty(t), (qi - 1) & 1))) return;
      ++(t ? nq1 : nq0);
      if (lane == 0) {
        if (x.q0 + t * kBM < 0) {
          mbar_arrive(bar_qfull(t));  // virtual tile: nothing to load
        } else {
          mbar_arrive_expect_tx(bar_qfull(t), C::kQBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(s_q + t * C::kQBytes + c * C::kChunkBytes, &tm_q, bar_qfull(t),
                        c * C::kChunkElems, x.q0 + t * kBM, x.b * p.Hq + x.h);
        }
      }
    };
    // One K or V tile into the next ring slot.  `zero_from` >= 0: a V tile
    // that holds key rows at or past the valid length L (those rows get
    // P = 0, but 0 * NaN is NaN, so they are zeroed before P V can read them;
    // a cache's unused tail may hold anything, rows past S are zero-filled
    // by TMA already).  That tile lands on a private barrier; this warp
    // zeroes the rows and then completes the slot's full barrier itself.
    auto load_kv = [&](const CUtensorMap* tm, int row, int bh_kv, int zero_from) {
      const int slot = ring % C::kSlots;
      if (ring >= C::kSlots && !(ok = wait_bar(bar_empty(slot), ((ring / C::kSlots) - 1) & 1)))
        return;
      const uint32_t dst = s_slots + slot * C::kTileBytes;
      const bool tail = zero_from >= 0;
      const uint32_t bar_land = tail ? bar_tail : bar_full(slot);
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_land, C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(dst + c * C::kChunkBytes, tm, bar_land, c * C::kChunkElems, row, bh_kv);
      }
      if (tail) {
        ok = wait_bar(bar_tail, ntail & 1);
        ++ntail;
        if (!ok) return;
        zero_rows_from<C::kChunks>(dst, zero_from, lane);
        if (lane == 0) mbar_arrive(bar_full(slot));
      }
      ++ring;
    };
    Item it, nx;
    int L = 0, n0 = 0, n1 = 0;
    bool have = next_item(it, L, n0, n1);
    bool early = false;  // Q_0 and K_0 of `it` went out with the previous item
    while (ok && have) {
      const int nm = max(n0, n1);
      const int bh_kv = it.b * p.Hkv + fast_div(it.h, p.div_G);
      const int j_tail = (L < p.S && (L & (kBN - 1)) != 0) ? L / kBN : -1;
      if (!early) load_q(it, 0);
      if (ok) load_q(it, 1);
      if (!ok) break;
      ++qi;
      int nL = 0, nn0 = 0, nn1 = 0;
      const bool have_nx = next_item(nx, nL, nn0, nn1);
      // With a causal diagonal (tile 1 visits one key tile more than tile 0)
      // the MMA warp starts the next item's tile 0 while tile 1 finishes
      // alone: that item's Q_0 and K_0 go out between this item's last K and
      // last V, the order the MMA warp consumes them.
      const bool early_next = have_nx && n0 >= 1 && n1 == n0 + 1;
      // K_0, V_0, K_1, V_1, ...: the order the MMA warp consumes them.
      for (int u = early ? 1 : 0; ok && u < 2 * nm; ++u) {
        if (u == 2 * nm - 1 && early_next) {
          load_q(nx, 0);
          if (ok) load_kv(&tm_k, 0, nx.b * p.Hkv + fast_div(nx.h, p.div_G), -1);
          if (!ok) break;
        }
        const bool is_v = u & 1;
        const int zero_from = (is_v && (u >> 1) == j_tail) ? (L & (kBN - 1)) : -1;
        load_kv(is_v ? &tm_v : &tm_k, (u >> 1) * kBN, bh_kv, zero_from);
      }
      it = nx;
      L = nL;
      n0 = nn0;
      n1 = nn1;
      have = have_nx;
      early = early_next;
    }
    // Drain: every issued copy must land before the CTA may exit (the last
    // kSlots ring entries cover every slot's latest copy).  Each Q buffer's
    // latest armed phase is waited for, which includes a next item's Q_0
    // issued early by a loop that then gave up on that item's K_0.
    for (int u = max(0, ring - C::kSlots); u < ring; ++u)
      mbar_wait(bar_full(u % C::kSlots), (u / C::kSlots) & 1, 3);
    if (nq0 > 0) mbar_wait(bar_qfull(0), (nq0 - 1) & 1, 3);
    if (nq1 > 0) mbar_wait(bar_qfull(1), (nq1 - 1) & 1, 3);
    if (ntail > 0) mbar_wait(bar_tail, (ntail - 1) & 1, 3);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp walks the schedule; one elected lane issues each
    // tcgen05 instruction.  Descriptors are built once per base address and
    // advanced by constants, so every MMA costs only its issue slot.
    constexpr uint32_t idesc_qk =
        kF8 ? idesc_e4m3(kBM, kBN, false, false) : idesc_f16kind(kBM, kBN, false, false, kF16);
    constexpr uint32_t idesc_pv =
        kF8 ? idesc_e4m3(kBM, D, false, true) : idesc_f16kind(kBM, D, false, true, kF16);
    const uint64_t dq0 = sdesc_sw128(s_q, 16, 1024);                // Q_0 as the A operand
    const uint64_t dk0 = sdesc_sw128(s_slots, 16, 1024);            // slot 0 as K (K-major B)
    const uint64_t dv0 = sdesc_sw128(s_slots, C::kChunkBytes, 1024);  // slot 0 as V (MN-major B)
    int ring = 0, qi = 0;
    uint32_t np0 = 0, np1 = 0;  // p_half waits so far, per tile
    bool ok = true;
    auto wait_slot = [&](int r) {
      const bool w = mbar_wait(bar_full(r % C::kSlots), (r / C::kSlots) & 1, 4, abort_flag);
      return __all_sync(0xffffffffu, w);
    };
    auto wait_bar = [&](uint32_t bar, uint32_t parity) {
      const bool w = mbar_wait(bar, parity, 6, abort_flag);
      return __all_sync(0xffffffffu, w);
    };
    // S_t = Q_t K^T for the K tile in `slot`.  The start-address field of a
    // descriptor is address >> 4 in its low 14 bits; shared addresses stay
    // below 2^18, so adding byte offsets >> 4 never carries out of it.
    auto issue_qk = [&](int t, int slot) {
      const uint64_t dq = dq0 + (uint64_t)((t * C::kQBytes) >> 4);
      const uint64_t dk = dk0 + (uint64_t)((slot * C::kTileBytes) >> 4);
#pragma unroll
      for (int kk = 0; kk < C::kKSteps; ++kk) {
        const uint32_t koff = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
        if constexpr (kF8)
          umma_ss_elect_f8(tmem + C::kColS(t), dq + koff, dk + koff, idesc_qk, kk > 0);
        else
          umma_ss_elect(tmem + C::kColS(t), dq + koff, dk + koff, idesc_qk, kk > 0);
      }
      umma_commit_elect(bar_s + 8 * t);
    };
    // O_t += P_t V for keys [64 * half, 64 * half + 64) of the tile in `slot`:
    // each step takes 32 bytes of P's row (8 TMEM columns) and 32 bytes' worth
    // of V rows (256 / EB bytes >> 4 further into the MN-major tile).
    auto issue_pv = [&](int t, int slot, int half, bool acc) {
      const uint64_t dv = dv0 + (uint64_t)((slot * C::kTileBytes) >> 4);
#pragma unroll
      for (int k4 = 0; k4 < C::kPvSteps; ++k4) {
        const int kk = half * C::kPvSteps + k4;
        const uint64_t bo = (uint64_t)(kk * (kF8 ? 256 : 128));
        if constexpr (kF8)
          umma_ts_elect_f8(tmem + C::kColO(t), tmem + C::kColS(t) + kk * 8, dv + bo, idesc_pv,
                           (acc || kk > 0) ? 1u : 0u);
        else
          umma_ts_elect(tmem + C::kColO(t), tmem + C::kColS(t) + kk * 8, dv + bo, idesc_pv,
                        (acc || kk > 0) ? 1u : 0u);
      }
    };
    // Next item with key tiles to visit and its tile counts (false when the
    // walk is over); the same sequence the load warp walks.
    auto next_item = [&](int& n0, int& n1) {
      Item x;
      while (unpack_item(sched_next<false>(sched, walk), x)) {
        const SeqGeom g = geom(p, x.b);
        n0 = tile_count(p, x.q0, g);
        n1 = tile_count(p, x.q0 + kBM, g);
        if (max(n0, n1) > 0) return true;
      }
      return false;
    };
    // S_t(0) of an item from its K_0 in `slot`; Q_t is read for the last time
    // when the tile visits at most one key tile.
    auto first_qk = [&](int t, int nt, int slot) {
      if (nt > 0) issue_qk(t, slot);
      if (nt <= 1) umma_commit_elect(bar_qempty(t));
    };
    int n0 = 0, n1 = 0;
    bool have = next_item(n0, n1);
    bool early = false;  // S_0(0) of the current item went out with the previous item
    int kslot0 = 0;      // ring slot of the current item's K_0
    while (ok && have) {
      const int nm = max(n0, n1);
      if (!early) {
        if (!(ok = wait_bar(bar_qfull(0), qi & 1))) break;
        kslot0 = ring % C::kSlots;
        if (!(ok = wait_slot(ring))) break;
        ++ring;
        tc_fence_after();
        first_qk(0, n0, kslot0);
      }
      if (!(ok = wait_bar(bar_qfull(1), qi & 1))) break;
      ++qi;
      tc_fence_after();
      first_qk(1, n1, kslot0);
      umma_commit_elect(bar_empty(kslot0));
      // The next item is walked after step 0's products are issued (the walk
      // costs this warp ~2000 cycles; there it overlaps the softmax of step 1).
      int nn0 = 0, nn1 = 0;
      bool have_nx = false, early_next = false;
      early = false;
      for (int j = 0; ok && j < nm; ++j) {
        const int vslot = ring % C::kSlots;
        if (!(ok = wait_slot(ring))) break;
        ++ring;
        const bool has_next = j + 1 < nm;
        bool next_ready = false;
        const int kslot = ring % C::kSlots;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < kQTiles; ++t) {
          const int nt = t ? n1 : n0;
          if (j >= nt) continue;
          uint32_t& npt = t ? np1 : np0;
          // P_t arrives in two halves; the first half's MMAs run while the
          // softmax group still computes the second.
          if (!(ok = wait_bar(bar_p + 16 * t, npt & 1))) break;
          tc_fence_after();
          issue_pv(t, vslot, 0, j > 0);
          if (!(ok = wait_bar(bar_p + 16 * t + 8, npt & 1))) break;
          ++npt;
          tc_fence_after();
          issue_pv(t, vslot, 1, true);
          if (j + 1 < nt) {
            if (!next_ready) {
              if (!(ok = wait_slot(ring))) break;
              next_ready = true;
              tc_fence_after();
            }
            issue_qk(t, kslot);
            if (j + 2 == nt) umma_commit_elect(bar_qempty(t));
          } else {
            umma_commit_elect(bar_o + 8 * t);  // O_t complete for this item
          }
        }
        if (!ok) break;
        umma_commit_elect(bar_empty(vslot));
        if (has_next) {
          // K_{j+1} is consumed by at least one tile because j + 1 < nm.
          umma_commit_elect(bar_empty(kslot));
          ++ring;
        }
        if (j == 0) {
          have_nx = next_item(nn0, nn1);
          // Causal diagonal: tile 1 visits one key tile more than tile 0.  Once
          // tile 0 is done (step n0 - 1) the next item's S_0(0) is issued from
          // its K_0, which the load warp placed between this item's last K and
          // V, so the tensor core is busy while tile 1 finishes alone.
          early_next = have_nx && n0 >= 1 && n1 == n0 + 1;
        }
        if (early_next && j == n0 - 1) {
          // Q_0 and K_0 of the next item (qi already counts this item)
          if (!(ok = wait_bar(bar_qfull(0), qi & 1))) break;
          kslot0 = ring % C::kSlots;
          if (!(ok = wait_slot(ring))) break;
          ++ring;
          tc_fence_after();
          first_qk(0, nn0, kslot0);
          early = true;
        }
      }
      n0 = nn0;
      n1 = nn1;
      have = have_nx;
    }
    // Drain: all issued MMAs complete before TMEM is released.
    umma_commit_elect(bar_drain);
    mbar_wait(bar_drain, 0, 7);
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int t = warp >> 2;                  // query tile of this group
    const int r = ((warp & 3) << 5) | lane;   // row within the tile = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t ts = lane_base + C::kColS(t);
    const uint32_t to = lane_base + C::kColO(t);
    const uint32_t bar_st = bar_s + 8 * t, bar_pt = bar_p + 16 * t, bar_ot = bar_o + 8 * t;
    const float sl2 = p.scale_log2;
    uint32_t ns = 0, no = 0;                  // s_full / o_full waits so far
    bool ok = true;

        Item it;
    while (ok && unpack_item(sched_next<false>(sched, walk), it)) {
      const SeqGeom sg = geom(p, it.b);
      const int L = sg.L, off = sg.off;
      const int q0t = it.q0 + t * kBM;
      const int n = tile_count(p, q0t, sg);
      const int i = q0t + r;
      const int pos = i + off;
      const bool row_ok = (i >= 0) && (i < p.T) && (i < sg.R);
      const int lim = p.causal ? min(L, pos + 1) : L;  // visible keys: [0, lim)
      float m_ref = -INFINITY;  // exponent reference (log2 units)
      float l = 0.f;

      for (int j = 0; j < n; ++j) {
        ok = mbar_wait(bar_st, ns & 1, 8, abort_flag);
        ++ns;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
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
        const bool masked = (k0 + kBN > L) || (p.causal && (k0 + kBN - 1 > q0t + off));
        if (masked) {
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (k0 + c >= lim) sr[c] = __float_as_uint(-INFINITY);
        }
        // Row maximum: eight independent chains of three-input max.
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
#pragma unroll
        for (int c = 0; c < kBN; c += 16) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            mx[e] = max3f(mx[e], __uint_as_float(sr[c + 2 * e]), __uint_as_float(sr[c + 2 * e + 1]));
        }
        const float m_tile =
            max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) *
            sl2;  // -inf stays -inf
        // Lazy rescale: move the reference only when the maximum ran ahead.
        const bool first = (m_ref == -INFINITY);
        const bool grow = !first && (m_tile > m_ref + kThresh);
        float alpha = 1.f;
        if (first && m_tile != -INFINITY) m_ref = m_tile;
        if (grow) {
          alpha = ex2_approx(m_ref - m_tile);
          l *= alpha;
          m_ref = m_tile;
        }

        // P = exp2(s * scale * log2e - m_ref), packed to bf16 pairs, in two
        // halves of 64 keys; each half is released to the MMA warp on its own.
        const float neg_ref = (m_ref == -INFINITY) ? 0.f : kPBias - m_ref;
        const float2 sl2x2 = make_float2(sl2, sl2);
        const float2 negx2 = make_float2(neg_ref, neg_ref);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0, acc2 = acc0, acc3 = acc0;
        uint32_t pk[kBN / 2];  // E4M3: the first kBN / 4 words
        float2 pprev = acc0;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int c = half * 64; c < half * 64 + 64; c += 8) {
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const float2 x = __ffma2_rn(
                  make_float2(__uint_as_float(sr[c + e]), __uint_as_float(sr[c + e + 1])), sl2x2,
                  negx2);
              const float2 pe = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              if constexpr (kF8) {
                if (e & 2) pk[(c + e) >> 2] = pack_e4m3x4(pprev.x, pprev.y, pe.x, pe.y);
                else pprev = pe;
              } else {
                pk[(c + e) >> 1] = pack2<kF16>(pe.x, pe.y);
              }
              if (e == 0) acc0 = __fadd2_rn(acc0, pe);
              else if (e == 2) acc1 = __fadd2_rn(acc1, pe);
              else if (e == 4) acc2 = __fadd2_rn(acc2, pe);
              else acc3 = __fadd2_rn(acc3, pe);
            }
          }
          if constexpr (kF8) tmem_st16(ts + 16 * half, pk + 16 * half);
          else tmem_st32(ts + 32 * half, pk + 32 * half);
          if (half == 0) {
            // O_t is final up to key tile j-1 here: PV_t(j-1) was issued
            // before S_t(j), whose completion this group has seen.  PV_t(j)
            // starts only after the arrive below, so it adds to the rescaled
            // row.
            if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
              for (int c = 0; c < D / 32; ++c) {
                uint32_t orr[32];
                tmem_ld32(to + 32 * c, orr);
                tmem_wait_ld32(orr);
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                tmem_st32(to + 32 * c, orr);
              }
            }
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar_pt + 8 * half);
        }
        const float2 s01 = __fadd2_rn(acc0, acc1), s23 = __fadd2_rn(acc2, acc3);
        const float2 s4 = __fadd2_rn(s01, s23);
        l += s4.x + s4.y;
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      if (n > 0) {
        ok = mbar_wait(bar_ot, no & 1, 9, abort_flag);
        ++no;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      const bool has = row_ok && (l > 0.f);
      const float inv = has ? p.o_scale / l : 0.f;
      uint16_t* orow =
          reinterpret_cast<uint16_t*>(p.o) + ((((size_t)it.b * p.Hq + it.h) * p.T) + i) * D;
      if (__any_sync(0xffffffffu, has)) {
        tc_fence_after();
        // 64 columns at a time; the next chunk's TMEM load is issued before
        // this chunk's stores so its latency overlaps them.
        uint32_t orr[64];
        tmem_ld32(to, orr);
        tmem_ld32(to + 32, orr + 32);
        tmem_wait_ld32(orr);
        tmem_wait_ld32(orr + 32);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t pkd[32];
#pragma unroll
          for (int e = 0; e < 32; ++e)
            pkd[e] = pack2<kF16>(__uint_as_float(orr[2 * e]) * inv,
                                 __uint_as_float(orr[2 * e + 1]) * inv);
          if (c + 1 < D / 64) {
            tmem_ld32(to + 64 * (c + 1), orr);
            tmem_ld32(to + 64 * (c + 1) + 32, orr + 32);
          }
          if (i >= 0 && i < p.T) {
            uint16_t* dst = orow + 64 * c;
            if (p.o_align32) {
#pragma unroll
              for (int v = 0; v < 4; ++v) st_global_v8(dst + 16 * v, pkd + 8 * v);
            } else {
#pragma unroll
              for (int v = 0; v < 8; ++v)
                reinterpret_cast<uint4*>(dst)[v] =
                    make_uint4(pkd[4 * v], pkd[4 * v + 1], pkd[4 * v + 2], pkd[4 * v + 3]);
            }
          }
          if (c + 1 < D / 64) {
            tmem_wait_ld32(orr);
            tmem_wait_ld32(orr + 32);
          }
        }
        tc_fence_before();
      } else if (i >= 0 && i < p.T) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
        for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0, 0, 0, 0);
      }
      if (p.lse != nullptr && i >= 0 && i < p.T) {
        p.lse[((size_t)it.b * p.Hq + it.h) * p.T + i] =
            has ? (m_ref - kPBias + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      }
    }
    // Items with no key tile: every row is padded (or past T): O = 0, LSE = -inf.
    while (ok && unpack_item(sched_next<true>(sched, walk + 1), it)) {
      const int i = it.q0 + t * kBM + r;
      if (i < 0 || i >= p.T) continue;
      const size_t row = ((size_t)it.b * p.Hq + it.h) * p.T + i;
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.o) + row * D);
#pragma unroll
      for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0, 0, 0, 0);
      if (p.lse != nullptr) p.lse[row] = -INFINITY;
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
