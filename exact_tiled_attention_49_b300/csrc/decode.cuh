// decode.cuh -- single-query KV-cache decode, split over the cache.
//
// "Implementing attention from scratch", KV caching: a decode step attends
// one new query over the S cached positions (the query sits at the last
// position, so the bottom-right causal mask admits every cached row), and
// decoding is bandwidth bound because every step reads the whole cache
// (Cost model).  Grouped-query attention lets the Hq / Hkv query heads of one
// KV head share a single read of its K and V rows.
//
// Pass 1 (decode_split_kernel): one block per (chunk of kChunk keys, kv head,
// sequence).  The block reads the chunk's K and V rows once for all G query
// heads of the group and reduces them to a partial result per head: the
// chunk maximum m (log2 units), denominator l and unnormalised output O.
// Pass 2 (decode_combine_kernel) merges the partials of every chunk with the
// online-softmax rescaling exp(m_chunk - m_max) ("Implementing attention from
// scratch", Stable softmax), normalises, and writes O and LSE.
#pragma once

#include "common.cuh"

namespace attn {
namespace decode {

constexpr int kChunk = 256;  // keys per split
constexpr int kWarps = 8;    // 32 keys per warp
constexpr int kThreads = kWarps * 32;

__host__ __device__ constexpr int max_splits(int S_max) { return (S_max + kChunk - 1) / kChunk; }

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
  int B, Hq, Hkv, S_max, splits;
  float scale_log2;     // scale * log2(e)
};

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

template <int DPL> struct Lanes;  // DPL consecutive elements of a row per lane

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

  // Scores: lane -> key.
  float s[G];
#pragma unroll
  for (int h = 0; h < G; ++h) s[h] = 0.f;
  const int j = w_begin + lane;
  if (lane < nk) {
    const uint4* kr = reinterpret_cast<const uint4*>(kbase + (size_t)j * D);
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
    load_lane<T, DPL>(vbase + (size_t)(w_begin + jj) * D, lane, vf);
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

// Merge the chunk partials of one (b, h): grid (Hq, B), D threads.
template <typename T, int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(Params p) {
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const int L = min(max(p.kv_lens[b], 0), p.S_max);
  const int n = (L + kChunk - 1) / kChunk;
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
  float M = -INFINITY;
  for (int s = 0; s < n; ++s) M = fmaxf(M, wm[s]);
  float acc = 0.f, l = 0.f;
  for (int s = 0; s < n; ++s) {
    const float sc = exp2f(wm[s] - M);
    acc = fmaf(sc, wo[(size_t)s * D + d], acc);
    l = fmaf(sc, wl[s], l);
  }
  store_out(o, acc / l);
  if (p.lse != nullptr && d == 0) p.lse[row] = (M + log2f(l)) * 0.69314718055994531f;
}

}  // namespace decode
}  // namespace attn
