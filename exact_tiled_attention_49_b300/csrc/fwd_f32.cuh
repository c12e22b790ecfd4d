// fwd_f32.cuh -- exact float32 prefill on the CUDA cores.
//
// The tiled method of "FlashAttention" (Transformers in Action, section
// 9.4.1, Figure 9.8) with the online softmax of "Implementing attention from
// scratch" (Core ideas, Stable softmax): each block owns BM query rows of one
// (batch, head), streams BN-key tiles of K and V through shared memory, and
// keeps per row a running maximum m, denominator l and unnormalised output;
// earlier sums are rescaled by exp(m_old - m_new) whenever m grows.  All
// arithmetic is float32 FFMA with the accurate expf (no TF32, no fast-math),
// for results within a few float32 ulps of the exact definition.
//
// Work split: 4 warps x 8 rows.  For one row, lane j scores key j of the
// tile (K rows padded to D+1 floats so the 32 lanes hit 32 banks), then the
// lanes switch to owning output columns d = lane + 32c for the P.V update.
#pragma once

#include "common.cuh"

namespace attn {
namespace f32fwd {

constexpr int kBM = 32;   // query rows per block
constexpr int kBN = 32;   // keys per tile (one per lane)
constexpr int kWarps = 4;
constexpr int kRowsPerWarp = kBM / kWarps;

struct Params {
  const float* q;
  const float* k;
  const float* v;
  float* o;
  float* lse;
  const int32_t* key_lens;
  const int32_t* q_pos;   // [B] key position of query row 0, or null (S - T)
  int B, Hq, Hkv, T, S, D;
  int causal;
  int k_off;              // global position of key row 0 (sharded keys; else 0)
  int shard;              // key_lens / q_pos are global positions (see seq_geom)
  float scale;
};

__host__ __device__ constexpr size_t smem_bytes(int D) {
  return sizeof(float) * ((size_t)kBM * D + (size_t)kBN * (D + 1) + (size_t)kBN * D);
}

// NC = number of 32-wide output column groups (D <= 32 * NC).
template <int NC>
__global__ void __launch_bounds__(kWarps * 32) fwd_f32_kernel(Params p) {
  extern __shared__ float smem[];
  const int D = p.D;
  float* q_s = smem;                       // [kBM][D]
  float* k_s = q_s + kBM * D;              // [kBN][D+1]
  float* v_s = k_s + kBN * (D + 1);        // [kBN][D]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (p.Hq / p.Hkv);
  const int q0 = blockIdx.x * kBM;
  // Row i sits at key position i + off: bottom-right (S - T) or, for chunked
  // prefill against a cache, q_pos[b]; keys below L are valid; rows below R
  // are not padded (common.cuh, seq_geom).
  const SeqGeom sg = seq_geom(p.key_lens, p.q_pos, p.k_off, p.shard != 0, b, p.T, p.S);
  const int off = sg.off, L = sg.L;

  const size_t q_base = (((size_t)b * p.Hq + h) * p.T) * D;
  const size_t kv_base = (((size_t)b * p.Hkv + g) * p.S) * D;

  for (int idx = threadIdx.x; idx < kBM * D; idx += blockDim.x) {
    const int r = idx / D, c = idx - r * D;
    q_s[idx] = (q0 + r < p.T) ? p.q[q_base + (size_t)(q0 + r) * D + c] : 0.f;
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][NC];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[r][c] = 0.f;
  }

  // Keys any row of this block can see.
  const int last_pos = q0 + kBM - 1 + off;
  const int kv_end = p.causal ? min(L, last_pos + 1) : L;

  for (int k0 = 0; k0 < kv_end; k0 += kBN) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kBN * D; idx += blockDim.x) {
      const int r = idx / D, c = idx - r * D;
      // Rows at or past L are never visible; they load as 0 so that a
      // cache's unused tail (which may hold anything) cannot reach P V.
      const bool in = (k0 + r) < L;
      const size_t gi = kv_base + (size_t)(k0 + r) * D + c;
      k_s[r * (D + 1) + c] = in ? p.k[gi] : 0.f;
      v_s[r * D + c] = in ? p.v[gi] : 0.f;
    }
    __syncthreads();

#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int rl = warp * kRowsPerWarp + r;
      const int i = q0 + rl;
      const int pos = i + off;
      const bool row_ok = (i < p.T) && (i < sg.R);
      const int j = k0 + lane;
      const bool vis = row_ok && (j < L) && (!p.causal || j <= pos);
      float s = -INFINITY;
      if (vis) {
        float dot = 0.f;
        const float* qr = q_s + rl * D;
        const float* kr = k_s + lane * (D + 1);
        for (int d = 0; d < D; ++d) dot = fmaf(qr[d], kr[d], dot);
        s = p.scale * dot;
      }
      const float m_new = fmaxf(m[r], warp_max(s));
      const float ref = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = expf(m[r] - ref);  // 0 while the row has seen nothing
      const float pj = vis ? expf(s - ref) : 0.f;
      l[r] = l[r] * alpha + warp_sum(pj);
      m[r] = m_new;
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[r][c] *= alpha;
      for (int jj = 0; jj < kBN; ++jj) {
        const float pb = __shfl_sync(0xffffffffu, pj, jj);
        if (pb != 0.f) {
          const float* vr = v_s + jj * D;
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const int d = lane + 32 * c;
            if (d < D) acc[r][c] = fmaf(pb, vr[d], acc[r][c]);
          }
        }
      }
    }
  }

#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int i = q0 + warp * kRowsPerWarp + r;
    if (i >= p.T) continue;
    const bool has = (l[r] > 0.f);
    const float inv = has ? 1.f / l[r] : 0.f;
    const size_t row = ((size_t)b * p.Hq + h) * p.T + i;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int d = lane + 32 * c;
      if (d < D) p.o[row * D + d] = has ? acc[r][c] * inv : 0.f;
    }
    if (p.lse != nullptr && lane == 0) p.lse[row] = has ? m[r] + logf(l[r]) : -INFINITY;
  }
}

}  // namespace f32fwd
}  // namespace attn
