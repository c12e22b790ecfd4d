// merge.cuh -- merge of attention partials computed over disjoint key sets.
//
// When the keys of a sequence are split into shards and each shard's
// attention is computed on its own (output O_n normalised over the shard,
// LSE_n = ln of the shard's sum of exponentials), the attention over all
// keys follows from the same rescaling the online softmax applies when its
// running maximum grows ("Implementing attention from scratch", Core ideas,
// Stable softmax; "Building a causal self-attention block from scratch in
// PyTorch", Extending It: sharding Q/K/V across devices and recombining):
//     LSE = ln sum_n exp(LSE_n),   O = sum_n exp(LSE_n - LSE) O_n.
// Two passes over a row's partials: their maximum M, then the sum in order
// n = 0, 1, ... with weights exp(LSE_n - M) <= 1, so no exponent overflows;
// a partial with LSE_n = -inf (its rows saw no key) adds nothing, and a row
// that no partial saw is O = 0, LSE = -inf.  The loads of one pass do not
// depend on each other, so a thread has all of a row's partials in flight
// at once (the merge is bound by memory, not arithmetic).
#pragma once

#include "common.cuh"

namespace attn {
namespace merge {

struct Params {
  const void* o_parts;     // [n_parts, rows, D] element type T
  const float* lse_parts;  // [n_parts, rows]
  void* o;                 // [rows, D] element type T
  float* lse;              // [rows] or null
  long long rows;
  int n_parts, D;
};

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kPer16B = 4;
  __device__ static void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  __device__ static uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};
template <bool kF16> struct Elem16 {
  static constexpr int kPer16B = 8;
  __device__ static void unpack(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = elem_lo<kF16>(w[i]);
      f[2 * i + 1] = elem_hi<kF16>(w[i]);
    }
  }
  __device__ static uint4 pack(const float* f) {
    return make_uint4(pack2<kF16>(f[0], f[1]), pack2<kF16>(f[2], f[3]), pack2<kF16>(f[4], f[5]),
                      pack2<kF16>(f[6], f[7]));
  }
};
template <> struct Elem<__nv_bfloat16> : Elem16<false> {};
template <> struct Elem<__half> : Elem16<true> {};

// One thread per 16 bytes of an output row; grid-stride over all of them.
template <typename T>
__global__ void __launch_bounds__(256) lse_merge_kernel(Params p) {
  using E = Elem<T>;
  constexpr int V = E::kPer16B;
  const int per_row = p.D / V;
  const long long total = p.rows * per_row;
  const uint4* parts = reinterpret_cast<const uint4*>(p.o_parts);
  uint4* out = reinterpret_cast<uint4*>(p.o);
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long row = idx / per_row;
    const int c = (int)(idx - row * per_row);
    float acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.f;
    float m = -INFINITY, l = 0.f;
#pragma unroll 4
    for (int n = 0; n < p.n_parts; ++n)  // NaN (never written) is ignored by fmaxf
      m = fmaxf(m, p.lse_parts[(long long)n * p.rows + row]);
    if (m > -INFINITY) {
#pragma unroll 4
      for (int n = 0; n < p.n_parts; ++n) {
        const float x = p.lse_parts[(long long)n * p.rows + row];
        // no key in this partial (or NaN): weight 0, and its O is not read
        const float w = (x > -INFINITY) ? expf(x - m) : 0.f;
        if (w > 0.f) {
          float f[V];
          E::unpack(parts[((long long)n * p.rows + row) * per_row + c], f);
#pragma unroll
          for (int e = 0; e < V; ++e) acc[e] = fmaf(w, f[e], acc[e]);
          l += w;
        }
      }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] *= inv;
    out[row * per_row + c] = E::pack(acc);
    if (p.lse != nullptr && c == 0) p.lse[row] = l > 0.f ? m + logf(l) : -INFINITY;
  }
}

}  // namespace merge
}  // namespace attn
