// decode.cuh -- single-query KV-cache decode, split over the cache.
//
// "Implementing attention from scratch", KV caching: a decode step attends
// one new query over the S cached positions (the query sits at the last
// position, so the bottom-right causal mask admits every cached row), and
// decoding is bandwidth bound because every step reads the whole cache
// (Cost model).  Grouped-query attention lets the G = Hq / Hkv query heads of
// one KV head share a single read of its K and V rows.
//
// Each (sequence, KV head) is a stream of cached keys.  Pieces of the streams
// are reduced independently to one partial result per query head: the
// piece's maximum m (log2 units), the denominator l and the unnormalised
// output O.
//   bf16: decode_split_mma_kernel -- persistent streaming warps on the tensor
//         cores (mma.sync m16n8k16), K/V streamed by TMA.  All streams, laid
//         end to end in 32-key sub-tiles, are cut into one contiguous,
//         equal span per warp, so every warp reads the same number of bytes
//         whatever the lengths; a warp carries its running softmax across
//         chunks and writes one partial per stream it touches.
//   fp32: decode_split_kernel -- one block per 256-key chunk on the CUDA
//         cores, exact float32 arithmetic.
// Pass 2 (decode_combine_spans_kernel, or decode_combine_kernel after the
// fp32 split) merges the partials of every piece with the
// online-softmax rescaling exp2(m_piece - m_max) ("Implementing attention
// from scratch", Stable softmax), normalises, and writes O and LSE.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace attn {
namespace decode {

constexpr int kChunk = 256;  // fp32 kernel: keys per block (one partial per chunk)
constexpr int kWarps = 8;    // fp32 kernel: 32 keys per warp
constexpr int kThreads = kWarps * 32;
constexpr int kSubKeys = 32;  // bf16 kernel: keys per sub-tile (the unit of the split)
constexpr int kMinSpan = 8;   // bf16 kernel: sub-tiles per warp at least (256 keys)

__host__ __device__ constexpr int max_splits(int S_max) { return (S_max + kChunk - 1) / kChunk; }

// Partial slots per (sequence, query head).  fp32: one per 256-key chunk.
// bf16: a stream of n <= ceil(S_max / 32) sub-tiles meets at most
// floor((n - 2) / 8) + 2 <= ceil(S_max / 256) + 1 spans of >= 8 sub-tiles.
__host__ __device__ constexpr int partial_slots(int S_max) { return max_splits(S_max) + 1; }

struct Params {
  const void* q;        // [B,Hq,D]
  const void* kc;       // [B,Hkv,S_max,D]
  const void* vc;       // [B,Hkv,S_max,D]
  const int32_t* kv_lens;
  void* o;              // [B,Hq,D]
  float* lse;           // [B,Hq] or null
  float* ws_o;          // [B,Hq,splits,D]
  float* ws_m;          // [B,Hq,splits]
  float* ws_l;          // [B,Hq,splits]
  long long* plan;      // bf16 split: [B + 2] prefix sums of sub-tiles per KV head,
                        // then the number of warps that took a span
  int B, Hq, Hkv, S_max, splits;  // splits = partial slots per (b, h)
  float scale_log2;     // scale * log2(e)
  // Fused append: the new token's K and V rows [B,Hkv,D], used for row
  // kv_len - 1 of each stream and written there, and the caches as
  // writable pointers.  Null: the caches are only read.
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  void* kc_w = nullptr;
  void* vc_w = nullptr;
};

// 32-key sub-tiles of a stream of L keys.
__device__ __forceinline__ int n_sub(int L) { return (L + kSubKeys - 1) / kSubKeys; }

// The span of stream keys (in sub-tiles) warp w of W takes: [w N / W, (w+1) N / W).
// The warp whose span holds sub-tile f is the largest w with w N / W <= f.
__device__ __forceinline__ long long span_begin(long long w, long long N, long long W) {
  return w * N / W;
}
__device__ __forceinline__ long long span_owner(long long f, long long N, long long W) {
  return ((f + 1) * W - 1) / N;
}

template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> { static constexpr int kPer16B = 8; };
template <> struct Vec<float> { static constexpr int kPer16B = 4; };

// Unpack a 16-byte vector into kPer16B floats.
__device__ __forceinline__ void unpack16(const uint4& u, float* f, __nv_bfloat16*) {
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}
__device__ __forceinline__ void unpack16(const uint4& u, float* f, float*) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T, int DPL>
__device__ __forceinline__ void load_lane(const T* row, int lane, float* f) {
#pragma unroll
  for (int e = 0; e < DPL; ++e) f[e] = to_f(row[lane * DPL + e]);
}
// Vectorised specialisations of the per-lane slice load.
template <>
__device__ __forceinline__ void load_lane<__nv_bfloat16, 4>(const __nv_bfloat16* row, int lane,
                                                            float* f) {
  const uint2 u = *reinterpret_cast<const uint2*>(row + lane * 4);
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
}
template <>
__device__ __forceinline__ void load_lane<__nv_bfloat16, 2>(const __nv_bfloat16* row, int lane,
                                                            float* f) {
  const uint32_t u = *reinterpret_cast<const uint32_t*>(row + lane * 2);
  f[0] = bf16_lo(u); f[1] = bf16_hi(u);
}
template <>
__device__ __forceinline__ void load_lane<float, 4>(const float* row, int lane, float* f) {
  const float4 u = *reinterpret_cast<const float4*>(row + lane * 4);
  f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w;
}
template <>
__device__ __forceinline__ void load_lane<float, 2>(const float* row, int lane, float* f) {
  const float2 u = *reinterpret_cast<const float2*>(row + lane * 2);
  f[0] = u.x; f[1] = u.y;
}

__device__ __forceinline__ void store_out(float* o, float x) { *o = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* o, float x) { *o = __float2bfloat16_rn(x); }
__device__ __forceinline__ void store_out(__half* o, float x) { *o = __float2half_rn(x); }

template <typename T, int D, int G>
__host__ __device__ constexpr size_t split_smem_bytes() {
  return sizeof(float) * ((size_t)D * G + 2 * (size_t)kWarps * G + (size_t)kWarps * G * D);
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(Params p) {
  constexpr int VEC = Vec<T>::kPer16B;
  constexpr int NV = D / VEC;   // 16-byte vectors per row
  constexpr int DPL = D / 32;   // output columns per lane
  extern __shared__ float smem[];
  float* q_s = smem;                        // [D][G], pre-scaled to log2 units
  float* red_m = q_s + D * G;               // [kWarps][G]
  float* red_l = red_m + kWarps * G;        // [kWarps][G]
  float* red_o = red_l + kWarps * G;        // [kWarps][G][D]

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int L = min(max(p.kv_lens[b], 0), p.S_max);
  const int k_begin = split * kChunk;
  if (k_begin >= L) return;  // nothing to read in this split
  const int k_end = min(L, k_begin + kChunk);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const T* qg = reinterpret_cast<const T*>(p.q) + ((size_t)b * p.Hq + (size_t)g * G) * D;
  for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
    const int h = idx / D, d = idx - h * D;
    q_s[d * G + h] = to_f(qg[idx]) * p.scale_log2;
  }
  __syncthreads();

  const size_t kv_row0 = ((size_t)b * p.Hkv + g) * p.S_max;
  const T* kbase = reinterpret_cast<const T*>(p.kc) + kv_row0 * D;
  const T* vbase = reinterpret_cast<const T*>(p.vc) + kv_row0 * D;
  const int w_begin = k_begin + warp * 32;
  const int nk = max(0, min(32, k_end - w_begin));
  // Fused append: row L - 1 is the new token; it is taken from k_new / v_new
  // (this warp alone reads that row in this launch) and written to the
  // caches below.
  const int jn = p.k_new != nullptr ? L - 1 : -1;
  const size_t new_row = ((size_t)b * p.Hkv + g) * D;

  // Scores: lane -> key.
  float s[G];
#pragma unroll
  for (int h = 0; h < G; ++h) s[h] = 0.f;
  const int j = w_begin + lane;
  if (lane < nk) {
    const uint4* kr = reinterpret_cast<const uint4*>(
        j == jn ? reinterpret_cast<const T*>(p.k_new) + new_row : kbase + (size_t)j * D);
#pragma unroll 4
    for (int c = 0; c < NV; ++c) {
      float kf[VEC];
      unpack16(__ldg(kr + c), kf, (T*)nullptr);
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float* qd = q_s + (c * VEC + e) * G;
#pragma unroll
        for (int h = 0; h < G; ++h) s[h] = fmaf(qd[h], kf[e], s[h]);
      }
    }
  } else {
#pragma unroll
    for (int h = 0; h < G; ++h) s[h] = -INFINITY;
  }

  // Warp-local softmax statistics per head.
  float pw[G], mw[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    mw[h] = warp_max(s[h]);
    pw[h] = (lane < nk) ? exp2f(s[h] - mw[h]) : 0.f;
    const float lw = warp_sum(pw[h]);
    if (lane == 0) {
      red_m[warp * G + h] = mw[h];
      red_l[warp * G + h] = lw;
    }
  }

  // P.V: lane -> DPL output columns, keys in order.
  float acc[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[h][e] = 0.f;
#pragma unroll 4
  for (int jj = 0; jj < nk; ++jj) {
    float vf[DPL];
    load_lane<T, DPL>(w_begin + jj == jn ? reinterpret_cast<const T*>(p.v_new) + new_row
                                         : vbase + (size_t)(w_begin + jj) * D,
                      lane, vf);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float pb = __shfl_sync(0xffffffffu, pw[h], jj);
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[h][e] = fmaf(pb, vf[e], acc[h][e]);
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < DPL; ++e) red_o[(warp * G + h) * D + lane * DPL + e] = acc[h][e];
  if (jn >= w_begin && jn < w_begin + nk) {
    const size_t dst = (kv_row0 + jn) * NV;
    for (int c = lane; c < NV; c += 32) {
      reinterpret_cast<uint4*>(p.kc_w)[dst + c] =
          reinterpret_cast<const uint4*>(p.k_new)[new_row / VEC + c];
      reinterpret_cast<uint4*>(p.vc_w)[dst + c] =
          reinterpret_cast<const uint4*>(p.v_new)[new_row / VEC + c];
    }
  }
  __syncthreads();

  // Merge the warps of this chunk into one partial per head.
  for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
    const int h = idx / D, d = idx - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * G + h]);
    float o = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mwv = red_m[w * G + h];
      const float sc = (mwv == -INFINITY) ? 0.f : exp2f(mwv - M);
      o = fmaf(sc, red_o[(w * G + h) * D + d], o);
      l = fmaf(sc, red_l[w * G + h], l);
    }
    const size_t slot = ((size_t)b * p.Hq + (size_t)g * G + h) * p.splits + split;
    p.ws_o[slot * D + d] = o;
    if (d == 0) {
      p.ws_m[slot] = M;
      p.ws_l[slot] = l;
    }
  }
}

// ---------------------------------------------------------------------------
// bf16 / fp16 pass 1: persistent streaming workers on the tensor cores.
//
// The streams of (sequence b, KV head g), in that order, are laid end to end
// as 32-key sub-tiles: stream (b, g) holds n_b = ceil(L_b / 32) of them and
// starts at sub-tile Hkv * P_b + g * n_b, P_b = n_0 + ... + n_{b-1}.  With N
// sub-tiles in all and W workers (warps), worker w takes the contiguous span
// [w N / W, (w + 1) N / W): every worker reads the same number of K/V bytes,
// give or take one sub-tile, whatever the lengths.  W is cut down to N / 8
// when the cache is small, so that every span holds >= 8 sub-tiles; a
// stream then meets at most ceil(S_max / 256) + 1 spans, which bounds the
// partial slots.  A worker carries its online softmax across the sub-tiles
// of one stream and writes one partial per stream it touches, into the slot
// numbered by its place among the workers that share that stream.  Every
// worker computes the prefix sums itself (one pass over the lengths); worker
// 0 also stores them, and the worker count, for the combine.
//
// A worker streams its span as 32-key sub-tiles through a private 2-stage
// ring: K and V arrive as 128B-swizzled TMA tiles (32 rows x 64 columns),
// the stream's q rows by a bulk copy when a stream starts, and the next
// sub-tile is in flight while one is computed.  Two stages leave room for 6
// workers per SM at D = 128 (3 stages: 4 workers, 2 in flight each), which
// measured faster: more workers beat more bytes in flight per worker.
//
// Per sub-tile: S = Q K^T with the G query heads as the M = 16 rows of
// mma.m16n8k16 (rows past G are zero) and K fragments from ldmatrix; the
// online softmax runs on the accumulator fragments (each thread holds 8
// scores of rows g and g + 8, the 4 threads of a row group finish the
// reductions with two shuffles); O += P V reuses the score fragments as the
// A operand (rounded to the input type), with V fragments from
// ldmatrix.trans.  Scores are scaled in fp32 (scale * log2 e) so that q keeps
// its exact input values.
struct Cursor {
  long long f;    // sub-tile index over all streams
  long long pb;   // P_b: sub-tiles per KV head of the sequences before b
  int b, g, j;    // sequence, KV head, sub-tile within the stream
  int n, L;       // sub-tiles and keys of sequence b's streams
  bool start;     // first sub-tile of a piece (stream start or span start)
};

__device__ __forceinline__ int seq_len(const Params& p, int b) {
  return min(max(__ldg(p.kv_lens + b), 0), p.S_max);
}

// Next sub-tile of the stream order (streams with no key are skipped).
__device__ __forceinline__ void cursor_next(const Params& p, Cursor& c) {
  ++c.f;
  c.start = false;
  if (++c.j < c.n) return;
  c.j = 0;
  c.start = true;
  if (++c.g < p.Hkv) return;
  c.g = 0;
  c.pb += c.n;
  for (++c.b; c.b < p.B; ++c.b) {
    c.L = seq_len(p, c.b);
    c.n = n_sub(c.L);
    if (c.n > 0) return;
  }
}

template <int D, int G>
struct MmaCfg {
  static constexpr int kSub = 32;                         // keys per sub-tile
  static constexpr int kStages = 2;
  static constexpr int kChunks = D / 64;                  // 128-byte column chunks
  static constexpr uint32_t kTileBytes = kSub * 128;      // one 32 x 64 box
  static constexpr uint32_t kKBytes = kChunks * kTileBytes;
  static constexpr uint32_t kStageBytes = 2 * kKBytes;    // K tiles then V tiles
  static constexpr uint32_t kQRawBytes = (uint32_t)G * D * 2;
  static constexpr uint32_t kQRawStride = (kQRawBytes + 127) / 128 * 128;
  static constexpr uint32_t kOffRing = 0;
  static constexpr uint32_t kOffQRaw = kOffRing + kStages * kStageBytes;
  static constexpr uint32_t kOffBars = kOffQRaw + 2 * kQRawStride;
  static constexpr uint32_t kWarpBytes = (kOffBars + 5 * 8 + 1023) / 1024 * 1024;
  static constexpr int kBudget = 220 * 1024;
  static constexpr int kWarps = (kBudget / kWarpBytes) > 8 ? 8 : (kBudget / kWarpBytes);
  static_assert(kWarps >= 1, "decode worker does not fit in shared memory");
  static constexpr size_t kSmemBytes = (size_t)kWarps * kWarpBytes + 1024;  // + alignment
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// d (16x8 fp32) += a (16x16, row) * b (16x8, col); a and b both bf16, or
// both fp16 when kF16.
template <bool kF16>
__device__ __forceinline__ void mma16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  if constexpr (kF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}
// Byte offset of 16-byte slot c (0..7) of row r in a 128B-swizzled tile.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// Inclusive prefix sum over the warp's lanes.
__device__ __forceinline__ long long warp_incl_scan(long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

// kF16: fp16 cache and query (else bf16).
template <int D, int G, bool kF16>
__global__ void __launch_bounds__(32 * MmaCfg<D, G>::kWarps)
    decode_split_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, Params p) {
  using C = MmaCfg<D, G>;
  constexpr int KS = D / 16;  // k-steps of Q K^T
  constexpr int NT = D / 8;   // n-tiles of P V
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem_all = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, tq = lane & 3;  // fragment row group, thread in the group
  uint8_t* smem = smem_all + warp * C::kWarpBytes;
  const uint32_t ring = smem_u32(smem + C::kOffRing);
  const uint32_t qraw = smem_u32(smem + C::kOffQRaw);
  const uint32_t bar_full = smem_u32(smem + C::kOffBars);  // [kStages]
  const uint32_t bar_q = bar_full + 8 * C::kStages;        // [2]

  if (lane == 0) {
    for (int i = 0; i < C::kStages + 2; ++i) mbar_init(bar_full + 8 * i, 1);
    fence_mbar_init();
  }
  __syncwarp();
  // Everything below may read what the previous kernel in the stream wrote.
  grid_dependency_wait();
  grid_dependents_launch();

  const int workers = gridDim.x * C::kWarps;
  const int worker = blockIdx.x * C::kWarps + warp;

  // Sub-tiles per KV head over all sequences (worker 0 stores the prefix
  // sums for the combine), then this worker's span.
  long long total = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    const long long n = b < p.B ? n_sub(seq_len(p, b)) : 0;
    const long long incl = warp_incl_scan(n, lane);
    if (worker == 0 && b < p.B) p.plan[b] = total + incl - n;
    total += __shfl_sync(0xffffffffu, incl, 31);
  }
  const long long N = total * p.Hkv;
  const long long W = min((long long)workers, max(1ll, N / kMinSpan));
  if (worker == 0 && lane == 0) {
    p.plan[p.B] = total;
    p.plan[p.B + 1] = W;
  }
  if (worker >= W || N == 0) return;
  const long long f_begin = span_begin(worker, N, W), f_end = span_begin(worker + 1, N, W);

  // Locate the first sub-tile: the sequence b whose streams hold f_begin.
  Cursor cc;
  {
    long long pre = 0;
    int found = -1;
    long long pb = 0;
    for (int b0 = 0; b0 < p.B && found < 0; b0 += 32) {
      const int b = b0 + lane;
      const long long n = b < p.B ? n_sub(seq_len(p, b)) : 0;
      const long long incl = warp_incl_scan(n, lane);
      const long long lo = (pre + incl - n) * p.Hkv, hi = (pre + incl) * p.Hkv;
      const uint32_t hit = __ballot_sync(0xffffffffu, n > 0 && lo <= f_begin && f_begin < hi);
      if (hit) {
        const int l = __ffs(hit) - 1;
        found = b0 + l;
        pb = __shfl_sync(0xffffffffu, pre + incl - n, l);
      }
      pre += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (found < 0) return;  // cannot happen for f_begin < N; keeps every read in range
    cc.b = found;
    cc.pb = pb;
    cc.L = seq_len(p, found);
    cc.n = n_sub(cc.L);
    const long long r = f_begin - pb * p.Hkv;
    cc.g = (int)(r / cc.n);
    cc.j = (int)(r - (long long)cc.g * cc.n);
    cc.f = f_begin;
    cc.start = true;
  }
  Cursor pf = cc;  // prefetch cursor, two sub-tiles ahead of the compute cursor
  int t_issue = 0, runs_issued = 0;

  auto issue = [&](const Cursor& c) {
    if (lane == 0) {
      const int row = (c.b * p.Hkv + c.g) * p.S_max + kSubKeys * c.j;
      const int st = t_issue % C::kStages;
      const uint32_t bar = bar_full + 8 * st;
      const uint32_t dst = ring + st * C::kStageBytes;
      mbar_arrive_expect_tx(bar, C::kStageBytes);
#pragma unroll
      for (int ch = 0; ch < C::kChunks; ++ch) {
        tma_load_2d(dst + ch * C::kTileBytes, &tm_k, bar, ch * 64, row);
        tma_load_2d(dst + C::kKBytes + ch * C::kTileBytes, &tm_v, bar, ch * 64, row);
      }
      if (c.start) {  // a new piece: its q rows too
        const int qb = runs_issued & 1;
        mbar_arrive_expect_tx(bar_q + 8 * qb, C::kQRawBytes);
        bulk_load(qraw + qb * C::kQRawStride,
                  reinterpret_cast<const uint16_t*>(p.q) +
                      ((size_t)c.b * p.Hq + (size_t)c.g * G) * D,
                  C::kQRawBytes, bar_q + 8 * qb);
      }
    }
    if (c.start) ++runs_issued;
    ++t_issue;
  };
  for (int k = 0; k < C::kStages - 1 && pf.f < f_end; ++k) {
    issue(pf);
    cursor_next(p, pf);
  }

  uint32_t qa[KS][4];        // Q fragments (rows = heads), fixed per piece
  float o[NT][4];            // O accumulator fragments
  float m_run[2], l_run[2];  // rows gr and gr + 8 (log2 units)
  int t = 0, run_seq = 0;
  bool ok = true;
  const float sl2 = p.scale_log2;
  while (cc.f < f_end && ok) {
    if (cc.start) {
      // new piece: Q fragments from its q rows; reset the running state
      const int qb = run_seq & 1;
      ok = mbar_wait(bar_q + 8 * qb, (run_seq >> 1) & 1, 0x29);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const uint8_t* qs = smem + C::kOffQRaw + qb * C::kQRawStride;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int c0 = ks * 16 + 2 * tq;
        qa[ks][0] = (gr < G) ? *reinterpret_cast<const uint32_t*>(qs + (gr * D + c0) * 2) : 0u;
        qa[ks][2] = (gr < G) ? *reinterpret_cast<const uint32_t*>(qs + (gr * D + c0 + 8) * 2) : 0u;
        qa[ks][1] = (gr + 8 < G)
                        ? *reinterpret_cast<const uint32_t*>(qs + ((gr + 8) * D + c0) * 2)
                        : 0u;
        qa[ks][3] = (gr + 8 < G)
                        ? *reinterpret_cast<const uint32_t*>(qs + ((gr + 8) * D + c0 + 8) * 2)
                        : 0u;
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
      m_run[0] = m_run[1] = -INFINITY;
      l_run[0] = l_run[1] = 0.f;
      ++run_seq;
      __syncwarp();
    }
    if (pf.f < f_end) {  // keep kStages - 1 sub-tiles in flight
      issue(pf);
      cursor_next(p, pf);
    }
    const int st = t % C::kStages;
    ok = mbar_wait(bar_full + 8 * st, (t / C::kStages) & 1, 0x2a);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    const int nkeys = min(kSubKeys, cc.L - kSubKeys * cc.j);
    const uint32_t kst = ring + st * C::kStageBytes;
    const uint32_t vst = kst + C::kKBytes;
    if (nkeys < kSubKeys) {
      // V rows past the sequence end may hold anything (NaN included): clear
      // them so that 0 * garbage cannot reach O
      uint8_t* vt = smem + C::kOffRing + st * C::kStageBytes + C::kKBytes;
      const int per_chunk = (kSubKeys - nkeys) * 8;
      for (int idx = lane; idx < per_chunk * C::kChunks; idx += 32) {
        const int ch = idx / per_chunk, rem = idx - ch * per_chunk;
        *reinterpret_cast<uint4*>(vt + ch * C::kTileBytes + (nkeys + rem / 8) * 128 +
                                  (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_shared();  // ordered before the copy that refills the stage
      __syncwarp();
    }
    if (p.k_new != nullptr && cc.j == (cc.L - 1) / kSubKeys) {
      // Fused append: the new token is the stream's last key, row L - 1.  Its
      // K and V rows replace what the copy brought for that row (the cache's
      // old contents) and go to the cache for later steps.  One 16-byte unit
      // per lane: D / 8 units of K, then D / 8 of V.  Only this worker reads
      // that row in this launch: every sub-tile belongs to one span.
      constexpr int kUnits = D / 8;
      const int r = (cc.L - 1) - kSubKeys * cc.j;
      if (lane < 2 * kUnits) {
        const bool isv = lane >= kUnits;
        const int u = isv ? lane - kUnits : lane;
        const size_t row = (size_t)cc.b * p.Hkv + cc.g;
        const uint4 val =
            reinterpret_cast<const uint4*>(isv ? p.v_new : p.k_new)[row * kUnits + u];
        uint8_t* tile = smem + C::kOffRing + st * C::kStageBytes + (isv ? C::kKBytes : 0u) +
                        (u >> 3) * C::kTileBytes;
        *reinterpret_cast<uint4*>(tile + sw128(r, u & 7)) = val;
        reinterpret_cast<uint4*>(isv ? p.vc_w : p.kc_w)[(row * p.S_max + (cc.L - 1)) * kUnits + u] =
            val;
      }
      fence_proxy_async_shared();  // ordered before the copy that refills the stage
      __syncwarp();
    }

    // S = Q K^T for the 32 keys: 4 n-tiles of 8 keys.
    float sacc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
      for (int u = 0; u < KS / 2; ++u) {
        // four 8x8 matrices: keys 8 nt .. 8 nt + 7, dims 32 u + 8 m
        const int m = lane >> 3, r = nt * 8 + (lane & 7), cg = 4 * u + m;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kst + (cg >> 3) * C::kTileBytes + sw128(r, cg & 7), b0, b1, b2, b3);
        mma16<kF16>(sacc[nt], qa[2 * u], b0, b1);
        mma16<kF16>(sacc[nt], qa[2 * u + 1], b2, b3);
      }
    }
    // Online softmax on the fragments: element e of n-tile nt is row
    // gr + 8 (e >> 1), key 8 nt + 2 tq + (e & 1).
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = nt * 8 + 2 * tq + (e & 1);
        const float x = (key < nkeys) ? sacc[nt][e] * sl2 : -INFINITY;
        sacc[nt][e] = x;
        mx[e >> 1] = fmaxf(mx[e >> 1], x);
      }
    }
    float alpha[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float mn = fmaxf(m_run[r], mx[r]);
      alpha[r] = (m_run[r] == -INFINITY) ? 0.f : ex2_approx(m_run[r] - mn);
      m_run[r] = mn;
      l_run[r] *= alpha[r];
    }
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][0] *= alpha[0];
        o[n][1] *= alpha[0];
        o[n][2] *= alpha[1];
        o[n][3] *= alpha[1];
      }
    }
    uint32_t pa[2][4];  // P as A fragments of the two 16-key k-steps
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float p0 = ex2_approx(sacc[nt][0] - m_run[0]);
      const float p1 = ex2_approx(sacc[nt][1] - m_run[0]);
      const float p2 = ex2_approx(sacc[nt][2] - m_run[1]);
      const float p3 = ex2_approx(sacc[nt][3] - m_run[1]);
      l_run[0] += p0 + p1;
      l_run[1] += p2 + p3;
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack2<kF16>(p0, p1);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack2<kF16>(p2, p3);
    }
    // O += P V: 2 k-steps of 16 keys, NT n-tiles of 8 output columns.
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
      for (int v = 0; v < NT / 2; ++v) {
        const int m = lane >> 3;
        const int r = ks * 16 + (m & 1) * 8 + (lane & 7), cg = 2 * v + (m >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vst + (cg >> 3) * C::kTileBytes + sw128(r, cg & 7), b0, b1, b2, b3);
        mma16<kF16>(o[2 * v], pa[ks], b0, b1);
        mma16<kF16>(o[2 * v + 1], pa[ks], b2, b3);
      }
    }
    __syncwarp();  // the stage may be refilled from here on

    if (cc.j + 1 == cc.n || cc.f + 1 == f_end) {
      // end of a piece: one partial per query head of the group, in the slot
      // numbered by this worker's place among the workers of the stream
      const long long s0 = cc.pb * p.Hkv + (long long)cc.g * cc.n;  // stream start
      const int slot = worker - (int)span_owner(s0, N, W);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float l = l_run[r];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        const int h = gr + 8 * r;
        if (h < G) {
          const size_t idx = ((size_t)cc.b * p.Hq + (size_t)cc.g * G + h) * p.splits + slot;
#pragma unroll
          for (int n = 0; n < NT; ++n)
            *reinterpret_cast<float2*>(p.ws_o + idx * D + n * 8 + 2 * tq) =
                make_float2(o[n][2 * r], o[n][2 * r + 1]);
          if (tq == 0) {
            p.ws_m[idx] = m_run[r];
            p.ws_l[idx] = l;
          }
        }
      }
    }
    cursor_next(p, cc);
    ++t;
  }
  // Drain: every issued copy has landed before the warp exits (immediate
  // unless a wait above timed out).
  if (lane == 0) {
    for (int k = 0; k < C::kStages; ++k) {
      const int tt = t_issue - 1 - k;
      if (tt >= 0) mbar_wait(bar_full + 8 * (tt % C::kStages), (tt / C::kStages) & 1, 0x2b);
    }
    for (int k = 0; k < 2; ++k) {
      const int ii = runs_issued - 1 - k;
      if (ii >= 0) mbar_wait(bar_q + 8 * (ii & 1), (ii >> 1) & 1, 0x2c);
    }
  }
}

// Merge the partials of the bf16 split kernel: one warp per (b, h), grid of
// ceil(B * Hq / 8) blocks of 8 warps.  The partials of (b, h) are the pieces
// of its stream, one per worker span that met it (found from the plan the
// split kernel stored), usually one to three: lane i reads piece i's
// maximum and denominator, the warp reduces them, and each lane then sums
// its D / 32 output columns over the pieces with 16-byte (D = 128) or
// 8-byte loads.  No block barrier and few dependent loads: the merge is
// latency bound, not bandwidth bound.
template <typename T, int D>
__global__ void __launch_bounds__(256) decode_combine_spans_kernel(Params p) {
  constexpr int C = D / 32;  // output columns per lane
  static_assert(C == 2 || C == 4, "D is 64 or 128");
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);  // b * Hq + h
  grid_dependency_wait();  // the partials and the plan come from the split kernel
  grid_dependents_launch();
  if (row >= (long long)p.B * p.Hq) return;
  const int b = (int)(row / p.Hq), h = (int)(row - (long long)b * p.Hq);
  const long long nb = p.plan[b + 1] - p.plan[b];  // sub-tiles of each stream of b
  int n = 0;
  if (nb > 0) {
    const long long N = p.plan[p.B] * p.Hkv, W = p.plan[p.B + 1];
    const long long s0 = p.plan[b] * p.Hkv + (long long)(h / (p.Hq / p.Hkv)) * nb;
    n = (int)(span_owner(s0 + nb - 1, N, W) - span_owner(s0, N, W)) + 1;
  }
  T* o = reinterpret_cast<T*>(p.o) + row * D + lane * C;
  if (n == 0) {
#pragma unroll
    for (int c = 0; c < C; ++c) store_out(o + c, 0.f);
    if (p.lse != nullptr && lane == 0) p.lse[row] = -INFINITY;
    return;
  }
  const float* wm = p.ws_m + row * p.splits;
  const float* wl = p.ws_l + row * p.splits;
  const float* wo = p.ws_o + row * p.splits * D + lane * C;
  // maximum over the pieces (n may exceed 32 for very long caches)
  float M = -INFINITY;
  for (int i = lane; i < n; i += 32) M = fmaxf(M, wm[i]);
  M = warp_max(M);
  float acc[C], l = 0.f;
#pragma unroll
  for (int c = 0; c < C; ++c) acc[c] = 0.f;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const float sc = i < n ? exp2f(wm[i] - M) : 0.f;
    l += i < n ? sc * wl[i] : 0.f;
    const int cnt = min(32, n - base);
    for (int k = 0; k < cnt; ++k) {
      const float w = __shfl_sync(0xffffffffu, sc, k);
      const float* src = wo + (size_t)(base + k) * D;
      if constexpr (C == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
        acc[2] = fmaf(w, v.z, acc[2]); acc[3] = fmaf(w, v.w, acc[3]);
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
      }
    }
  }
  l = warp_sum(l);
  const float inv = 1.f / l;
#pragma unroll
  for (int c = 0; c < C; ++c) store_out(o + c, acc[c] * inv);
  if (p.lse != nullptr && lane == 0) p.lse[row] = (M + log2f(l)) * 0.69314718055994531f;
}

// The same merge with one block of 8 warps per (b, h), for launches whose
// streams are few and long (one sequence of 131k tokens: ~111 pieces per
// stream), where one warp per head would leave most SMs idle and walk its
// pieces one by one: warp w takes pieces w, w + 8, ... against the row's
// maximum M, and the block adds the 8 partial sums.
template <typename T, int D>
__global__ void __launch_bounds__(256) decode_combine_heads_kernel(Params p) {
  constexpr int C = D / 32;  // output columns per lane
  static_assert(C == 2 || C == 4, "D is 64 or 128");
  __shared__ float red_o[8][D];
  __shared__ float red_x[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = blockIdx.x;  // b * Hq + h
  grid_dependency_wait();  // the partials and the plan come from the split kernel
  grid_dependents_launch();
  const int b = (int)(row / p.Hq), h = (int)(row - (long long)b * p.Hq);
  const long long nb = p.plan[b + 1] - p.plan[b];  // sub-tiles of each stream of b
  int n = 0;
  if (nb > 0) {
    const long long N = p.plan[p.B] * p.Hkv, W = p.plan[p.B + 1];
    const long long s0 = p.plan[b] * p.Hkv + (long long)(h / (p.Hq / p.Hkv)) * nb;
    n = (int)(span_owner(s0 + nb - 1, N, W) - span_owner(s0, N, W)) + 1;
  }
  T* o = reinterpret_cast<T*>(p.o) + row * D;
  if (n == 0) {
    for (int d = threadIdx.x; d < D; d += blockDim.x) store_out(o + d, 0.f);
    if (p.lse != nullptr && threadIdx.x == 0) p.lse[row] = -INFINITY;
    return;
  }
  const float* wm = p.ws_m + row * p.splits;
  const float* wl = p.ws_l + row * p.splits;
  const float* wo = p.ws_o + row * p.splits * D + lane * C;
  float M = -INFINITY;
  for (int i = threadIdx.x; i < n; i += blockDim.x) M = fmaxf(M, wm[i]);
  M = warp_max(M);
  if (lane == 0) red_x[warp] = M;
  __syncthreads();
  M = red_x[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) M = fmaxf(M, red_x[w]);
  __syncthreads();  // red_x is reused below
  float acc[C], l = 0.f;
#pragma unroll
  for (int c = 0; c < C; ++c) acc[c] = 0.f;
  for (int i = warp; i < n; i += 8) {
    const float sc = exp2f(wm[i] - M);
    l = fmaf(sc, wl[i], l);
    const float* src = wo + (size_t)i * D;
    if constexpr (C == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] = fmaf(sc, v.x, acc[0]); acc[1] = fmaf(sc, v.y, acc[1]);
      acc[2] = fmaf(sc, v.z, acc[2]); acc[3] = fmaf(sc, v.w, acc[3]);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src);
      acc[0] = fmaf(sc, v.x, acc[0]); acc[1] = fmaf(sc, v.y, acc[1]);
    }
  }
#pragma unroll
  for (int c = 0; c < C; ++c) red_o[warp][lane * C + c] = acc[c];
  if (lane == 0) red_x[warp] = l;
  __syncthreads();
  float lt = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) lt += red_x[w];
  const float inv = 1.f / lt;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float x = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) x += red_o[w][d];
    store_out(o + d, x * inv);
  }
  if (p.lse != nullptr && threadIdx.x == 0) p.lse[row] = (M + log2f(lt)) * 0.69314718055994531f;
}

// Merge the chunk partials of the fp32 split kernel (one per 256-key chunk)
// of one (b, h): grid (Hq, B), D threads.
template <typename T, int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(Params p) {
  __shared__ float sc_s[1024];
  __shared__ float red[D / 32];
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  grid_dependency_wait();  // the partials come from the split kernel
  grid_dependents_launch();
  const int Lb = min(max(p.kv_lens[b], 0), p.S_max);
  const int n = (Lb + kChunk - 1) / kChunk;  // partials to merge, from slot 0
  const size_t row = (size_t)b * p.Hq + h;
  T* o = reinterpret_cast<T*>(p.o) + row * D + d;
  if (n == 0) {
    store_out(o, 0.f);
    if (p.lse != nullptr && d == 0) p.lse[row] = -INFINITY;
    return;
  }
  const float* wm = p.ws_m + row * p.splits;
  const float* wl = p.ws_l + row * p.splits;
  const float* wo = p.ws_o + row * p.splits * D;
  float acc = 0.f, l = 0.f, M = -INFINITY;
  for (int base = 0; base < n; base += 1024) {
    const int cnt = min(1024, n - base);
    // maximum of this batch of partial maxima, block-wide
    float mloc = -INFINITY;
    for (int s = d; s < cnt; s += D) mloc = fmaxf(mloc, wm[base + s]);
    mloc = warp_max(mloc);
    if ((d & 31) == 0) red[d >> 5] = mloc;
    __syncthreads();
    float Mb = -INFINITY;
#pragma unroll
    for (int w = 0; w < D / 32; ++w) Mb = fmaxf(Mb, red[w]);
    const float Mn = fmaxf(M, Mb);
    const float r = (M == -INFINITY) ? 0.f : exp2f(M - Mn);
    acc *= r;
    l *= r;
    M = Mn;
    for (int s = d; s < cnt; s += D) sc_s[s] = exp2f(wm[base + s] - M);
    __syncthreads();
#pragma unroll 8
    for (int s = 0; s < cnt; ++s) {
      const float sc = sc_s[s];
      acc = fmaf(sc, wo[(size_t)(base + s) * D + d], acc);
      l = fmaf(sc, wl[base + s], l);
    }
    __syncthreads();
  }
  store_out(o, acc / l);
  if (p.lse != nullptr && d == 0) p.lse[row] = (M + log2f(l)) * 0.69314718055994531f;
}

}  // namespace decode
}  // namespace attn
