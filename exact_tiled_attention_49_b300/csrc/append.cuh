// append.cuh -- KV-cache append: one new token's K and V rows per
// (batch, kv head) written at cache position pos[b].
//
// "Building a causal self-attention block from scratch in PyTorch", Step 5
// appends each new token along the sequence axis of the cache;
// "Implementing attention from scratch", KV caching, places it at offset
// "cache length".  The cache here is preallocated to S_max positions, so the
// append is a bounds-checked row copy with 128-bit loads and stores.
#pragma once

#include "common.cuh"

namespace attn {

// One thread per 16-byte vector; grid-stride over B * Hkv * vec_per_row.
__global__ void __launch_bounds__(256)
    kv_append_kernel(uint4* __restrict__ kc, uint4* __restrict__ vc,
                     const uint4* __restrict__ kn, const uint4* __restrict__ vn,
                     const int32_t* __restrict__ pos, int B, int Hkv, int S_max,
                     int vec_per_row, int* dev_status) {
  const long long total = (long long)B * Hkv * vec_per_row;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long bg = idx / vec_per_row;
    const int c = (int)(idx - bg * vec_per_row);
    const int b = (int)(bg / Hkv);
    const int p = pos[b];
    if (p < 0 || p >= S_max) {
      if (c == 0 && dev_status != nullptr) atomicOr(dev_status, 1);
      continue;
    }
    const long long dst = (bg * S_max + p) * vec_per_row + c;
    kc[dst] = kn[idx];
    vc[dst] = vn[idx];
  }
}

}  // namespace attn
