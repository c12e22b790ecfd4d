// bwd_f32.cuh -- attention backward (dQ, dK, dV) in exact float32 on the CUDA
// cores, the counterpart of the fp32 forward (fwd_f32.cuh): FFMA, accurate
// expf, no TF32.
//
// The chain rule through the softmax ("Hands-on build guide:
// FlashAttention-style tiled attention kernel in pure NumPy", Roadmap:
// gradient through attention), with the weights recomputed from the
// forward's LSE ("Self-Attention: Implementation, Complexity, and Efficient
// Variants", FlashAttention: the backward recomputes the attention matrix):
//   P = exp(scale q_i . k_j - LSE_i) on visible (i, j), dP = dO_i . v_j,
//   dS = P (dP - delta_i), delta_i = dO_i . O_i,
//   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i
// (query heads of a GQA group summed into their KV head).
//
//   bwd_f32_delta_kernel   one warp per query row: delta.
//   bwd_f32_dq_kernel      one warp per query row: lane = key for the two dot
//                          products of 32 keys at a time, lane = output
//                          column for dQ += dS k_j (rows read whole).
//   bwd_f32_dkdv_kernel    one warp per key row, over the query rows of every
//                          head of its group: lane = query row for the dots,
//                          lane = column for dK and dV.
// Rows past the valid key length are never read (they may hold anything);
// padded rows and rows that see no key get dQ = 0 and add nothing.  A
// correctness path: it reads K, V (dQ) or Q, dO (dK/dV) once per row.
#pragma once

#include "common.cuh"

namespace attn {
namespace f32bwd {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct Params {
  const float* q;           // [B,Hq,T,D]
  const float* k;           // [B,Hkv,S,D]
  const float* v;           // [B,Hkv,S,D]
  const float* o;           // [B,Hq,T,D]
  const float* dout;        // [B,Hq,T,D]
  const float* lse;         // [B,Hq,T]
  float* delta;             // [B,Hq,T] workspace
  float* dq;                // [B,Hq,T,D]
  float* dk;                // [B,Hkv,S,D]
  float* dv;                // [B,Hkv,S,D]
  const int32_t* key_lens;  // [B] or null
  const int32_t* q_pos;     // [B] or null (S - T)
  int B, Hq, Hkv, T, S, D, causal;
  float scale;
};

// Valid keys L and the key position of query row 0 (both clamped as in the
// forward kernels).
__device__ __forceinline__ int f32_key_bound(const Params& p, int b) {
  return p.key_lens != nullptr ? min(max(p.key_lens[b], 0), p.S) : p.S;
}
__device__ __forceinline__ int f32_q_offset(const Params& p, int b) {
  return p.q_pos != nullptr ? min(max(p.q_pos[b], -(p.T + 256)), p.S) : p.S - p.T;
}

// delta[row] = dO[row] . O[row]
__global__ void __launch_bounds__(kThreads) bwd_f32_delta_kernel(Params p, long long rows) {
  const long long row = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* orow = p.o + row * p.D;
  const float* drow = p.dout + row * p.D;
  float acc = 0.f;
  for (int d = lane; d < p.D; d += 32) acc = fmaf(orow[d], drow[d], acc);
  acc = warp_sum(acc);
  if (lane == 0) p.delta[row] = acc;
}

// One warp per query row (b, h, i); NC = ceil(D / 32) output columns per lane.
template <int NC>
__global__ void __launch_bounds__(kThreads) bwd_f32_dq_kernel(Params p) {
  extern __shared__ float smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * kWarps + warp, h = blockIdx.y, b = blockIdx.z;
  if (i >= p.T) return;
  const int D = p.D;
  float* q_s = smem + warp * 2 * D;  // this row's q and dO
  float* do_s = q_s + D;
  const size_t row = ((size_t)b * p.Hq + h) * p.T + i;
  const int g = h / (p.Hq / p.Hkv);
  const int L = f32_key_bound(p, b), off = f32_q_offset(p, b);
  const int pos = i + off;
  // visible keys [0, lim); none for a padded row
  const int lim = (pos >= L) ? 0 : max(0, p.causal ? min(L, pos + 1) : L);
  float acc[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] = 0.f;
  if (lim > 0) {
    for (int d = lane; d < D; d += 32) {
      q_s[d] = p.q[row * D + d];
      do_s[d] = p.dout[row * D + d];
    }
    __syncwarp();
    const float lse = p.lse[row], dlt = p.delta[row];
    const float* kb = p.k + ((size_t)b * p.Hkv + g) * p.S * D;
    const float* vb = p.v + ((size_t)b * p.Hkv + g) * p.S * D;
    for (int j0 = 0; j0 < lim; j0 += 32) {
      const int j = j0 + lane;
      float ds = 0.f;
      if (j < lim) {
        const float* kr = kb + (size_t)j * D;
        const float* vr = vb + (size_t)j * D;
        float s = 0.f, dp = 0.f;
        for (int d = 0; d < D; ++d) {
          s = fmaf(q_s[d], kr[d], s);
          dp = fmaf(do_s[d], vr[d], dp);
        }
        const float pr = expf(s * p.scale - lse);
        ds = pr * (dp - dlt);
      }
      const int nk = min(32, lim - j0);
      for (int jj = 0; jj < nk; ++jj) {
        const float dsj = __shfl_sync(0xffffffffu, ds, jj);
        const float* kr = kb + (size_t)(j0 + jj) * D;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int d = lane + 32 * c;
          if (d < D) acc[c] = fmaf(dsj, kr[d], acc[c]);
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int d = lane + 32 * c;
    if (d < D) p.dq[row * D + d] = acc[c] * p.scale;
  }
}

// One warp per key row (b, g, j), over the query rows of the G heads of
// group g; NC = ceil(D / 32) output columns per lane.
template <int NC>
__global__ void __launch_bounds__(kThreads) bwd_f32_dkdv_kernel(Params p) {
  extern __shared__ float smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x * kWarps + warp, g = blockIdx.y, b = blockIdx.z;
  if (j >= p.S) return;
  const int D = p.D;
  const int G = p.Hq / p.Hkv;
  float* k_s = smem + warp * 2 * D;  // this key's k and v
  float* v_s = k_s + D;
  const size_t krow = ((size_t)b * p.Hkv + g) * p.S + j;
  const int L = f32_key_bound(p, b), off = f32_q_offset(p, b);
  float ak[NC], av[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) ak[c] = av[c] = 0.f;
  if (j < L) {
    for (int d = lane; d < D; d += 32) {
      k_s[d] = p.k[krow * D + d];
      v_s[d] = p.v[krow * D + d];
    }
    __syncwarp();
    // query rows that see key j: i + off >= j (causal), i + off < L (not
    // padded), 0 <= i < T
    const int i_lo = p.causal ? max(0, j - off) : 0;
    const int i_hi = min(p.T, L - off);
    for (int hh = 0; hh < G; ++hh) {
      const int h = g * G + hh;
      const size_t rbase = ((size_t)b * p.Hq + h) * p.T;
      for (int i0 = i_lo; i0 < i_hi; i0 += 32) {
        const int i = i0 + lane;
        float pr = 0.f, ds = 0.f;
        if (i < i_hi) {
          const float* qr = p.q + (rbase + i) * D;
          const float* dr = p.dout + (rbase + i) * D;
          float s = 0.f, dp = 0.f;
          for (int d = 0; d < D; ++d) {
            s = fmaf(qr[d], k_s[d], s);
            dp = fmaf(dr[d], v_s[d], dp);
          }
          pr = expf(s * p.scale - p.lse[rbase + i]);
          ds = pr * (dp - p.delta[rbase + i]);
        }
        const int nq = min(32, i_hi - i0);
        for (int ii = 0; ii < nq; ++ii) {
          const float pi = __shfl_sync(0xffffffffu, pr, ii);
          const float dsi = __shfl_sync(0xffffffffu, ds, ii);
          const float* qr = p.q + (rbase + i0 + ii) * D;
          const float* dr = p.dout + (rbase + i0 + ii) * D;
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const int d = lane + 32 * c;
            if (d < D) {
              av[c] = fmaf(pi, dr[d], av[c]);
              ak[c] = fmaf(dsi, qr[d], ak[c]);
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int d = lane + 32 * c;
    if (d < D) {
      p.dk[krow * D + d] = ak[c] * p.scale;
      p.dv[krow * D + d] = av[c];
    }
  }
}

}  // namespace f32bwd
}  // namespace attn
