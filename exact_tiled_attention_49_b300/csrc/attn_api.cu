// attn_api.cu -- host side of libattn.so: argument validation, TMA tensor-map
// encoding and kernel dispatch behind the C ABI declared in include/attn.h.
//
// Everything is one translation unit so that the device error word and the
// kernels need no relocatable device code.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <utility>
#include <vector>

#include "../../include/attn.h"
#include "append.cuh"
#include "bwd_bf16_tc.cuh"
#include "bwd_f32.cuh"
#include "common.cuh"
#include "decode.cuh"
#include "fwd_bf16_tc.cuh"
#include "fwd_f32.cuh"
#include "merge.cuh"

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxDevices = 64;

std::atomic<unsigned long long> g_launches{0};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// cuTensorMapEncodeTiled from the driver, resolved once through the runtime.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 3-D 16-bit tensor [outer, rows, D] (D contiguous; bf16, or fp16 when f16)
// loaded as boxes of 64 columns x 128 rows with 128-byte swizzle; rows past
// `rows` read as 0.
bool make_tmap_bf16(CUtensorMap* m, const void* base, int D, int rows, long long outer,
                    bool f16 = false) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)rows * (cuuint64_t)D * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D 8-bit tensor [outer, rows, D] (D = 128 contiguous, E4M3 bytes) loaded
// as boxes of 128 columns x 128 rows with 128-byte swizzle.
bool make_tmap_u8(CUtensorMap* m, const void* base, int D, int rows, long long outer) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)D, (cuuint64_t)rows * (cuuint64_t)D};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D 16-bit tensor [rows, D] (D contiguous; bf16, or fp16 when f16) loaded
// as boxes of 64 columns x `box_rows` rows with 128-byte swizzle.
bool make_tmap_bf16_2d(CUtensorMap* m, const void* base, int D, long long rows, int box_rows,
                       bool f16 = false) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Opt a kernel into more than 48 KB of dynamic shared memory, once per device.
template <typename K>
bool ensure_smem(K kernel, size_t bytes, std::atomic<uint64_t>& done_mask) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  const uint64_t bit = 1ull << dev;
  if (done_mask.load(std::memory_order_acquire) & bit) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
      cudaSuccess)
    return false;
  // Ask for the largest shared-memory carveout so that as many CTAs as the
  // shared-memory budget allows can be resident on one SM.
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return false;
  done_mask.fetch_or(bit, std::memory_order_acq_rel);
  return true;
}

// Streaming-multiprocessor count of the current device (cached per device).
int num_sms() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
    v = 148;
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

// Launch as a programmatic dependent of the previous kernel in the stream: the
// kernel's CTAs may be scheduled while that kernel drains and wait in
// hardware (griddepcontrol.wait) before touching its results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

int launch_status() {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaPeekAtLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// ------------------------------------------------------------- prefill

// kF8: E4M3 inputs with per-tensor descales (qkv_descale), bf16 output.
template <int D, bool kF16, bool kF8 = false>
int launch_fwd_tc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                  int Hq, int Hkv, int T, int S, int causal, const int32_t* key_lens,
                  const int32_t* q_pos, float scale, cudaStream_t st,
                  const float* qkv_descale = nullptr, int k_off = 0, bool shard = false) {
  using namespace attn::tcfwd;
  using C = Cfg<D, kF8 ? 1 : 2>;
  static std::atomic<uint64_t> smem_done{0};
  auto kernel = fwd_bf16_tc_kernel<D, kF16, kF8>;
  if (!ensure_smem(kernel, C::kSmemAlloc, smem_done)) return ATTN_ERR_CUDA;
  CUtensorMap tq, tk, tv;
  if constexpr (kF8) {
    if (!make_tmap_u8(&tq, q, D, T, (long long)B * Hq) ||
        !make_tmap_u8(&tk, k, D, S, (long long)B * Hkv) ||
        !make_tmap_u8(&tv, v, D, S, (long long)B * Hkv))
      return ATTN_ERR_CUDA;
  } else {
    if (!make_tmap_bf16(&tq, q, D, T, (long long)B * Hq, kF16) ||
        !make_tmap_bf16(&tk, k, D, S, (long long)B * Hkv, kF16) ||
        !make_tmap_bf16(&tv, v, D, S, (long long)B * Hkv, kF16))
      return ATTN_ERR_CUDA;
  }
  Params p;
  p.o = o;
  p.lse = lse;
  p.key_lens = key_lens;
  p.q_pos = q_pos;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.T = T;
  p.S = S;
  p.causal = causal ? 1 : 0;
  p.k_off = k_off;
  p.shard = shard ? 1 : 0;
  // Pair slots per (batch, head): a sequence whose count of query tiles
  // with a non-padded row is odd has its pairs shifted 128 rows down, so it
  // needs room for T + 128 rows.  Without key_lens and q_pos every sequence
  // has ceil(T / 128) such tiles.
  const int shift_all = (((T + kBM - 1) / kBM) & 1) ? kBM : 0;
  const int span = (key_lens != nullptr || q_pos != nullptr) ? T + kBM : T + shift_all;
  p.n_pairs = (span + kItemRows - 1) / kItemRows;
  const long long items = (long long)p.n_pairs * B * Hq;
  if (items >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
  p.n_items = (int)items;
  p.o_align32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
  p.div_B = attn::make_fast_div((uint32_t)B);
  p.div_Hq = attn::make_fast_div((uint32_t)Hq);
  p.div_G = attn::make_fast_div((uint32_t)(Hq / Hkv));
  p.scale_log2 = scale * kLog2e;
  p.o_scale = 1.f;
  if constexpr (kF8) {
    p.scale_log2 = scale * qkv_descale[0] * qkv_descale[1] * kLog2e;
    p.o_scale = qkv_descale[2];
  }
  // Persistent: one CTA per SM (the kernel takes all 512 TMEM columns).
  const int grid = (int)std::min<long long>(num_sms(), items);
  kernel<<<grid, kThreads, C::kSmemAlloc, st>>>(tq, tk, tv, p);
  return launch_status();
}

template <int NC>
int launch_fwd_f32(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int Hq, int Hkv, int T, int S, int D, int causal, const int32_t* key_lens,
                   const int32_t* q_pos, float scale, cudaStream_t st, int k_off, bool shard) {
  using namespace attn::f32fwd;
  static std::atomic<uint64_t> smem_done{0};
  auto kernel = fwd_f32_kernel<NC>;
  const size_t smem = smem_bytes(D);
  if (!ensure_smem(kernel, smem_bytes(32 * NC), smem_done)) return ATTN_ERR_CUDA;
  Params p;
  p.q = static_cast<const float*>(q);
  p.k = static_cast<const float*>(k);
  p.v = static_cast<const float*>(v);
  p.o = static_cast<float*>(o);
  p.lse = lse;
  p.key_lens = key_lens;
  p.q_pos = q_pos;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.T = T;
  p.S = S;
  p.D = D;
  p.causal = causal ? 1 : 0;
  p.k_off = k_off;
  p.shard = shard ? 1 : 0;
  p.scale = scale;
  dim3 grid((T + kBM - 1) / kBM, Hq, B);
  kernel<<<grid, kWarps * 32, smem, st>>>(p);
  return launch_status();
}

// ------------------------------------------------------------- backward

template <int D, bool kF16>
int launch_bwd_tc(const attn::tcbwd::Params& p0, const void* q, const void* k, const void* v,
                  const void* dout, cudaStream_t st) {
  using namespace attn::tcbwd;
  static std::atomic<uint64_t> smem_dq{0}, smem_dkdv{0};
  auto kdq = bwd_dq_kernel<D, kF16>;
  auto kdkdv = bwd_dkdv_kernel<D, kF16>;
  if (!ensure_smem(kdq, Cfg<D>::kSmemAlloc, smem_dq) ||
      !ensure_smem(kdkdv, Cfg<D>::kSmemAlloc, smem_dkdv))
    return ATTN_ERR_CUDA;
  CUtensorMap tq, tdo, tk, tv;
  if (!make_tmap_bf16(&tq, q, D, p0.T, (long long)p0.B * p0.Hq, kF16) ||
      !make_tmap_bf16(&tdo, dout, D, p0.T, (long long)p0.B * p0.Hq, kF16) ||
      !make_tmap_bf16(&tk, k, D, p0.S, (long long)p0.B * p0.Hkv, kF16) ||
      !make_tmap_bf16(&tv, v, D, p0.S, (long long)p0.B * p0.Hkv, kF16))
    return ATTN_ERR_CUDA;
  const long long rows = (long long)p0.B * p0.Hq * p0.T;
  const long long rows_per_block = 8 * (32 / (D / 8));  // 8 warps, 32 / (D / 8) rows each
  const long long want_blocks = (rows + rows_per_block - 1) / rows_per_block;
  const unsigned blocks = (unsigned)std::min<long long>(want_blocks, (long long)num_sms() * 16);
  bwd_delta_kernel<kF16><<<blocks, 256, 0, st>>>(p0, rows);
  int rc = launch_status();
  if (rc != ATTN_OK) return rc;
  // x = (batch, head) varies fastest, so the heaviest tiles of every head
  // are dispatched first
  kdq<<<dim3(p0.B * p0.Hq, p0.n_qtiles), kThreads, Cfg<D>::kSmemAlloc, st>>>(tq, tdo, tk, tv, p0);
  rc = launch_status();
  if (rc != ATTN_OK) return rc;
  kdkdv<<<dim3(p0.B * p0.Hkv, p0.n_ktiles), kThreads, Cfg<D>::kSmemAlloc, st>>>(tq, tdo, tk, tv,
                                                                               p0);
  return launch_status();
}

// Exact fp32 backward (bwd_f32.cuh): any 1 <= D <= 256, 4-byte alignment.
template <int NC>
int launch_bwd_f32(const attn::f32bwd::Params& p, cudaStream_t st) {
  using namespace attn::f32bwd;
  const size_t smem = (size_t)kWarps * 2 * p.D * sizeof(float);
  bwd_f32_dq_kernel<NC><<<dim3((p.T + kWarps - 1) / kWarps, p.Hq, p.B), kThreads, smem, st>>>(p);
  int rc = launch_status();
  if (rc != ATTN_OK) return rc;
  bwd_f32_dkdv_kernel<NC><<<dim3((p.S + kWarps - 1) / kWarps, p.Hkv, p.B), kThreads, smem, st>>>(p);
  return launch_status();
}

int bwd_f32(const void* q, const void* k, const void* v, const void* o, const void* dout,
            const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int T, int S,
            int D, int causal, const int32_t* key_lens, const int32_t* q_pos, float scale,
            void* workspace, size_t ws_bytes, attn_stream_t stream) {
  if (D > 256) return ATTN_ERR_UNSUPPORTED;
  if (!aligned4(q) || !aligned4(k) || !aligned4(v) || !aligned4(o) || !aligned4(dout) ||
      !aligned4(dq) || !aligned4(dk) || !aligned4(dv) || !aligned4(lse) ||
      (key_lens != nullptr && !aligned4(key_lens)) || (q_pos != nullptr && !aligned4(q_pos)))
    return ATTN_ERR_INVALID_ARG;
  const size_t need = ((size_t)B * Hq * T * sizeof(float) + 15) / 16 * 16;
  if (workspace == nullptr || ws_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
  attn::f32bwd::Params p{};
  p.q = static_cast<const float*>(q);
  p.k = static_cast<const float*>(k);
  p.v = static_cast<const float*>(v);
  p.o = static_cast<const float*>(o);
  p.dout = static_cast<const float*>(dout);
  p.lse = lse;
  p.delta = static_cast<float*>(workspace);
  p.dq = static_cast<float*>(dq);
  p.dk = static_cast<float*>(dk);
  p.dv = static_cast<float*>(dv);
  p.key_lens = key_lens;
  p.q_pos = q_pos;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.T = T;
  p.S = S;
  p.D = D;
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const long long rows = (long long)B * Hq * T;
  attn::f32bwd::bwd_f32_delta_kernel<<<(unsigned)((rows + attn::f32bwd::kWarps - 1) /
                                                  attn::f32bwd::kWarps),
                                       attn::f32bwd::kThreads, 0, st>>>(p, rows);
  const int rc = launch_status();
  if (rc != ATTN_OK) return rc;
  switch ((D + 31) / 32) {
    case 1: return launch_bwd_f32<1>(p, st);
    case 2: return launch_bwd_f32<2>(p, st);
    case 3: return launch_bwd_f32<3>(p, st);
    case 4: return launch_bwd_f32<4>(p, st);
    case 5: return launch_bwd_f32<5>(p, st);
    case 6: return launch_bwd_f32<6>(p, st);
    case 7: return launch_bwd_f32<7>(p, st);
    default: return launch_bwd_f32<8>(p, st);
  }
}

// -------------------------------------------------------------- decode

template <typename T, int D, int G>
int launch_decode_g(const attn::decode::Params& p, cudaStream_t st) {
  using namespace attn::decode;
  if constexpr (!std::is_same<T, float>::value) {
    // bf16 / fp16: persistent tensor-core workers, one CTA per SM at most
    constexpr bool kF16 = std::is_same<T, __half>::value;
    using C = MmaCfg<D, G>;
    static std::atomic<uint64_t> smem_done{0};
    auto kernel = decode_split_mma_kernel<D, G, kF16>;
    if (!ensure_smem(kernel, C::kSmemBytes, smem_done)) return ATTN_ERR_CUDA;
    const long long rows = (long long)p.B * p.Hkv * p.S_max;
    if (rows + kSubKeys >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
    CUtensorMap tk, tv;
    if (!make_tmap_bf16_2d(&tk, p.kc, D, rows, C::kSub, kF16) ||
        !make_tmap_bf16_2d(&tv, p.vc, D, rows, C::kSub, kF16))
      return ATTN_ERR_CUDA;
    // Persistent: one CTA per SM at most, enough warps that every warp's
    // span can hold >= kMinSpan sub-tiles when the cache is full.
    const long long subtiles = (long long)p.B * p.Hkv * ((p.S_max + kSubKeys - 1) / kSubKeys);
    const long long want = (subtiles / kMinSpan + C::kWarps - 1) / C::kWarps;
    const long long ctas = std::max<long long>(1, std::min<long long>(num_sms(), want));
    launch_pdl(kernel, dim3((unsigned)ctas), dim3(32 * C::kWarps), C::kSmemBytes, st, tk, tv, p);
    if (launch_status() != ATTN_OK) return ATTN_ERR_CUDA;
    const long long heads = (long long)p.B * p.Hq;
    if ((long long)p.B * p.Hkv * 8 < ctas * C::kWarps)
      // few, long streams (more than ~8 pieces each): a block per head
      launch_pdl(decode_combine_heads_kernel<T, D>, dim3((unsigned)heads), dim3(256), 0, st, p);
    else  // one warp per head
      launch_pdl(decode_combine_spans_kernel<T, D>, dim3((unsigned)((heads + 7) / 8)), dim3(256),
                 0, st, p);
    return launch_status();
  } else {
    // fp32: one block per (chunk, kv head, sequence) on the CUDA cores
    static std::atomic<uint64_t> smem_done{0};
    auto kernel = decode_split_kernel<T, D, G>;
    constexpr size_t smem = split_smem_bytes<T, D, G>();
    if (!ensure_smem(kernel, smem, smem_done)) return ATTN_ERR_CUDA;
    kernel<<<dim3(p.splits, p.Hkv, p.B), kThreads, smem, st>>>(p);
  }
  int rc = launch_status();
  if (rc != ATTN_OK) return rc;
  launch_pdl(decode_combine_kernel<T, D>, dim3(p.Hq, p.B), dim3(D), 0, st, p);
  return launch_status();
}

template <typename T, int D>
int launch_decode_d(const attn::decode::Params& p, int G, cudaStream_t st) {
  switch (G) {
    case 1: return launch_decode_g<T, D, 1>(p, st);
    case 2: return launch_decode_g<T, D, 2>(p, st);
    case 4: return launch_decode_g<T, D, 4>(p, st);
    case 8: return launch_decode_g<T, D, 8>(p, st);
    case 16: return launch_decode_g<T, D, 16>(p, st);
    default: return ATTN_ERR_UNSUPPORTED;
  }
}

bool finite_positive(float x) { return std::isfinite(x) && x > 0.f; }

// The size, type and scale rules of the prefill (what fwd_dispatch checks
// before any launch, pointers aside).
int fwd_check_sizes(int B, int Hq, int Hkv, int T, int S, int D, int dtype, float scale) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || S <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !finite_positive(scale)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_F16 && dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (dtype != ATTN_F32 && D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (dtype == ATTN_F32 && D > 256) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// Device layout of attn_fwd_host's workspace: q, k, v, o, lse and key_lens
// at 256-byte aligned offsets.
struct HostLayout {
  size_t q, k, v, o, lse, lens, total;
};
inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }
HostLayout host_layout(int B, int Hq, int Hkv, int T, int S, int D, int dtype) {
  const size_t es = dtype == ATTN_F32 ? 4 : 2;
  const size_t nq = (size_t)B * Hq * T * D * es, nk = (size_t)B * Hkv * S * D * es;
  HostLayout l;
  l.q = 0;
  l.k = align256(nq);
  l.v = l.k + align256(nk);
  l.o = l.v + align256(nk);
  l.lse = l.o + align256(nq);
  l.lens = l.lse + align256((size_t)B * Hq * T * sizeof(float));
  l.total = l.lens + align256((size_t)B * sizeof(int32_t));
  return l;
}

// attn_fwd_host's pipeline stages: ranges of (sequence, KV head) groups,
// either whole sequences [b0, b0 + nb) (ng = Hkv) or KV heads [g0, g0 + ng)
// of one sequence (nb = 1), so that each stage's q, k, v, o and lse are
// contiguous.  About 32 MiB of inputs per stage, at most 16 stages per
// sequence range.
struct HostChunk {
  int b0, nb, g0, ng;
};
std::vector<HostChunk> host_chunks(int B, int Hkv, size_t in_bytes) {
  constexpr size_t kStageBytes = 32u << 20;
  const long long units = (long long)B * Hkv;
  const long long want = std::min<long long>(16, std::max<long long>(1, (long long)((in_bytes + kStageBytes - 1) / kStageBytes)));
  const long long per = (units + want - 1) / want;
  std::vector<HostChunk> out;
  if (per >= Hkv) {
    const int nb = (int)((per + Hkv - 1) / Hkv);
    for (int b = 0; b < B; b += nb) out.push_back({b, std::min(nb, B - b), 0, Hkv});
  } else {
    for (int b = 0; b < B; ++b)
      for (int g = 0; g < Hkv; g += (int)per) out.push_back({b, 1, g, std::min((int)per, Hkv - g)});
  }
  return out;
}

// Shared by attn_fwd, attn_fwd_chunked and attn_fwd_kv_shard: validation and
// kernel choice.  `shard`: key_lens and q_pos are global positions and the
// keys start at global position k_off (common.cuh, seq_geom).
int fwd_dispatch(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                 int Hq, int Hkv, int T, int S, int D, int dtype, int causal,
                 const int32_t* key_lens, const int32_t* q_pos, float scale,
                 attn_stream_t stream, int k_off = 0, bool shard = false) {
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || S <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !finite_positive(scale)) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (lse != nullptr && !aligned4(lse)) return ATTN_ERR_INVALID_ARG;
  if (key_lens != nullptr && !aligned4(key_lens)) return ATTN_ERR_INVALID_ARG;
  if (q_pos != nullptr && !aligned4(q_pos)) return ATTN_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == ATTN_BF16 || dtype == ATTN_F16) {
    if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
      return ATTN_ERR_INVALID_ARG;
    const bool f16 = dtype == ATTN_F16;
#define ATTN_TC_CASE(DD, F)                                                                  \
  return launch_fwd_tc<DD, F>(q, k, v, o, lse, B, Hq, Hkv, T, S, causal, key_lens, q_pos, \
                              scale, st, nullptr, k_off, shard);
    if (D == 64) {
      if (f16) ATTN_TC_CASE(64, true) else ATTN_TC_CASE(64, false)
    }
    if (f16) ATTN_TC_CASE(128, true) else ATTN_TC_CASE(128, false)
#undef ATTN_TC_CASE
  }
  if (dtype == ATTN_F32) {
    if (D > 256) return ATTN_ERR_UNSUPPORTED;
    if (!aligned4(q) || !aligned4(k) || !aligned4(v) || !aligned4(o)) return ATTN_ERR_INVALID_ARG;
    const int nc = (D + 31) / 32;
#define ATTN_F32_CASE(N)                                                                    \
  case N:                                                                                   \
    return launch_fwd_f32<N>(q, k, v, o, lse, B, Hq, Hkv, T, S, D, causal, key_lens, q_pos, \
                             scale, st, k_off, shard);
    switch (nc) {
      ATTN_F32_CASE(1) ATTN_F32_CASE(2) ATTN_F32_CASE(3) ATTN_F32_CASE(4)
      ATTN_F32_CASE(5) ATTN_F32_CASE(6) ATTN_F32_CASE(7) ATTN_F32_CASE(8)
      default: return ATTN_ERR_UNSUPPORTED;
    }
#undef ATTN_F32_CASE
  }
  return ATTN_ERR_INVALID_ARG;
}

}  // namespace

namespace attn {
// One warp waits on a barrier that no thread arrives at: the bounded wait
// must give up, record its site in the error word and let the kernel return.
__global__ void selftest_wait_kernel() {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, 0xEE, &abort_flag);
  __syncwarp();
}
}  // namespace attn

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int T, int S, int D, int dtype, int causal, const int32_t* key_lens,
             float scale, attn_stream_t stream) {
  return fwd_dispatch(q, k, v, o, lse, B, Hq, Hkv, T, S, D, dtype, causal, key_lens, nullptr,
                      scale, stream);
}

size_t attn_fwd_host_workspace_size(int B, int Hq, int Hkv, int T, int S, int D, int dtype) {
  if (fwd_check_sizes(B, Hq, Hkv, T, S, D, dtype, 1.f) != ATTN_OK) return 0;
  return host_layout(B, Hq, Hkv, T, S, D, dtype).total;
}

int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                  int Hkv, int T, int S, int D, int dtype, int causal, const int32_t* key_lens,
                  float scale, void* workspace, size_t ws_bytes, attn_stream_t stream,
                  attn_stream_t copy_in, attn_stream_t copy_out) {
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  const int rc0 = fwd_check_sizes(B, Hq, Hkv, T, S, D, dtype, scale);
  if (rc0 != ATTN_OK) return rc0;
  const HostLayout lay = host_layout(B, Hq, Hkv, T, S, D, dtype);
  if (workspace == nullptr || ws_bytes < lay.total || !aligned16(workspace))
    return ATTN_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t cin = copy_in ? reinterpret_cast<cudaStream_t>(copy_in) : st;
  cudaStream_t cout = copy_out ? reinterpret_cast<cudaStream_t>(copy_out) : st;
  char* ws = static_cast<char*>(workspace);
  char *dq = ws + lay.q, *dk = ws + lay.k, *dv = ws + lay.v, *dout = ws + lay.o;
  float* dlse = reinterpret_cast<float*>(ws + lay.lse);
  int32_t* dlens = key_lens != nullptr ? reinterpret_cast<int32_t*>(ws + lay.lens) : nullptr;
  const size_t es = dtype == ATTN_F32 ? 4 : 2;
  const int G = Hq / Hkv;
  const size_t in_bytes = lay.k + 2 * (lay.v - lay.k);
  const std::vector<HostChunk> chunks = host_chunks(B, Hkv, in_bytes);
  const int n = (int)chunks.size();

  // Events: fork, one "inputs in" and one "computed" per chunk, join.
  std::vector<cudaEvent_t> ev(2 * n + 2, nullptr);
  auto release = [&]() {
    for (cudaEvent_t e : ev)
      if (e != nullptr) cudaEventDestroy(e);  // freed once the event completes
  };
  for (auto& e : ev)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
      e = nullptr;
      release();
      return ATTN_ERR_CUDA;
    }
  cudaEvent_t fork = ev[0], join = ev[2 * n + 1];
  auto ev_in = [&](int c) { return ev[1 + c]; };
  auto ev_done = [&](int c) { return ev[1 + n + c]; };
  bool ok = cudaEventRecord(fork, st) == cudaSuccess &&
            cudaStreamWaitEvent(cin, fork, 0) == cudaSuccess &&
            cudaStreamWaitEvent(cout, fork, 0) == cudaSuccess;
  if (ok && dlens != nullptr)
    ok = cudaMemcpyAsync(dlens, key_lens, (size_t)B * sizeof(int32_t), cudaMemcpyHostToDevice,
                         cin) == cudaSuccess;
  // Byte offsets of a chunk in the [B, H, rows, D] layouts.
  auto q_off = [&](const HostChunk& c) { return ((size_t)c.b0 * Hq + (size_t)c.g0 * G) * T * D * es; };
  auto q_len = [&](const HostChunk& c) { return (size_t)c.nb * c.ng * G * T * D * es; };
  auto k_off = [&](const HostChunk& c) { return ((size_t)c.b0 * Hkv + c.g0) * S * D * es; };
  auto k_len = [&](const HostChunk& c) { return (size_t)c.nb * c.ng * S * D * es; };
  auto l_off = [&](const HostChunk& c) { return ((size_t)c.b0 * Hq + (size_t)c.g0 * G) * T; };
  auto l_len = [&](const HostChunk& c) { return (size_t)c.nb * c.ng * G * T; };
  // Enqueued phase by phase (all copies in, all launches, all copies out),
  // so that a copy to pageable host memory, which returns only when it is
  // done, cannot hold back the enqueueing of the other chunks.
  for (int c = 0; ok && c < n; ++c) {
    const HostChunk& ch = chunks[c];
    ok = cudaMemcpyAsync(dq + q_off(ch), static_cast<const char*>(q) + q_off(ch), q_len(ch),
                         cudaMemcpyHostToDevice, cin) == cudaSuccess &&
         cudaMemcpyAsync(dk + k_off(ch), static_cast<const char*>(k) + k_off(ch), k_len(ch),
                         cudaMemcpyHostToDevice, cin) == cudaSuccess &&
         cudaMemcpyAsync(dv + k_off(ch), static_cast<const char*>(v) + k_off(ch), k_len(ch),
                         cudaMemcpyHostToDevice, cin) == cudaSuccess &&
         cudaEventRecord(ev_in(c), cin) == cudaSuccess;
  }
  int rc = ok ? ATTN_OK : ATTN_ERR_CUDA;
  for (int c = 0; rc == ATTN_OK && c < n; ++c) {
    const HostChunk& ch = chunks[c];
    if (cudaStreamWaitEvent(st, ev_in(c), 0) != cudaSuccess) {
      rc = ATTN_ERR_CUDA;
      break;
    }
    rc = fwd_dispatch(dq + q_off(ch), dk + k_off(ch), dv + k_off(ch), dout + q_off(ch),
                      lse != nullptr ? dlse + l_off(ch) : nullptr, ch.nb, ch.ng * G, ch.ng, T, S,
                      D, dtype, causal, dlens != nullptr ? dlens + ch.b0 : nullptr, nullptr, scale,
                      stream);
    if (rc == ATTN_OK && cudaEventRecord(ev_done(c), st) != cudaSuccess) rc = ATTN_ERR_CUDA;
  }
  for (int c = 0; rc == ATTN_OK && c < n; ++c) {
    const HostChunk& ch = chunks[c];
    if (cudaStreamWaitEvent(cout, ev_done(c), 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<char*>(o) + q_off(ch), dout + q_off(ch), q_len(ch),
                        cudaMemcpyDeviceToHost, cout) != cudaSuccess ||
        (lse != nullptr &&
         cudaMemcpyAsync(lse + l_off(ch), dlse + l_off(ch), l_len(ch) * sizeof(float),
                         cudaMemcpyDeviceToHost, cout) != cudaSuccess))
      rc = ATTN_ERR_CUDA;
  }
  // Join: work enqueued on `stream` after this call follows the last copy out.
  if (cudaEventRecord(join, cout) != cudaSuccess || cudaStreamWaitEvent(st, join, 0) != cudaSuccess)
    rc = ATTN_ERR_CUDA;
  release();
  return rc;
}

int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int T, int S, int D, int causal, const int32_t* key_lens, float scale,
                 float q_descale, float k_descale, float v_descale, attn_stream_t stream) {
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || S <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !finite_positive(scale) || !finite_positive(q_descale) ||
      !finite_positive(k_descale) || !finite_positive(v_descale))
    return ATTN_ERR_INVALID_ARG;
  if (D != 128 || B > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr && !aligned4(lse)) return ATTN_ERR_INVALID_ARG;
  if (key_lens != nullptr && !aligned4(key_lens)) return ATTN_ERR_INVALID_ARG;
  const float descale[3] = {q_descale, k_descale, v_descale};
  return launch_fwd_tc<128, false, true>(q, k, v, o, lse, B, Hq, Hkv, T, S, causal, key_lens,
                                         nullptr, scale, reinterpret_cast<cudaStream_t>(stream),
                                         descale);
}

int attn_fwd_chunked(const void* q, const void* kcache, const void* vcache, void* o, float* lse,
                     const int32_t* q_pos, const int32_t* kv_lens, int B, int Hq, int Hkv,
                     int T, int S_max, int D, int dtype, int causal, float scale,
                     attn_stream_t stream) {
  if (!q_pos || !kv_lens) return ATTN_ERR_INVALID_ARG;
  return fwd_dispatch(q, kcache, vcache, o, lse, B, Hq, Hkv, T, S_max, D, dtype, causal, kv_lens,
                      q_pos, scale, stream);
}

int attn_fwd_kv_shard(const void* q, const void* k, const void* v, void* o, float* lse,
                      const int32_t* q_pos, const int32_t* key_lens, int k_off, int B, int Hq,
                      int Hkv, int T, int S, int D, int dtype, int causal, float scale,
                      attn_stream_t stream) {
  if (!q_pos || !key_lens || k_off < 0) return ATTN_ERR_INVALID_ARG;
  if (k_off >= (1 << 30) || T >= (1 << 30) || S >= (1 << 30)) return ATTN_ERR_UNSUPPORTED;
  return fwd_dispatch(q, k, v, o, lse, B, Hq, Hkv, T, S, D, dtype, causal, key_lens, q_pos,
                      scale, stream, k_off, true);
}

int attn_lse_merge(const void* o_parts, const float* lse_parts, int n_parts, void* o, float* lse,
                   int B, int Hq, int T, int D, int dtype, attn_stream_t stream) {
  if (!o_parts || !lse_parts || !o) return ATTN_ERR_INVALID_ARG;
  if (n_parts <= 0 || B <= 0 || Hq <= 0 || T <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  size_t esz;
  if (dtype == ATTN_BF16 || dtype == ATTN_F16) esz = 2;
  else if (dtype == ATTN_F32) esz = 4;
  else return ATTN_ERR_INVALID_ARG;
  if ((size_t)D * esz % 16 != 0 || D > 1024) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(o_parts) || !aligned16(o) || !aligned4(lse_parts) ||
      (lse != nullptr && !aligned4(lse)))
    return ATTN_ERR_INVALID_ARG;
  attn::merge::Params p;
  p.o_parts = o_parts;
  p.lse_parts = lse_parts;
  p.o = o;
  p.lse = lse;
  p.rows = (long long)B * Hq * T;
  p.n_parts = n_parts;
  p.D = D;
  const long long threads = p.rows * (long long)((size_t)D * esz / 16);
  const long long blocks = std::max<long long>(
      1, std::min<long long>((threads + 255) / 256, (long long)num_sms() * 16));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == ATTN_BF16)
    attn::merge::lse_merge_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(p);
  else if (dtype == ATTN_F16)
    attn::merge::lse_merge_kernel<__half><<<(unsigned)blocks, 256, 0, st>>>(p);
  else
    attn::merge::lse_merge_kernel<float><<<(unsigned)blocks, 256, 0, st>>>(p);
  return launch_status();
}

size_t attn_bwd_workspace_size(int B, int Hq, int T) {
  if (B <= 0 || Hq <= 0 || T <= 0) return 0;
  return ((size_t)B * Hq * T * sizeof(float) + 15) / 16 * 16;
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int T, int S,
             int D, int dtype, int causal, const int32_t* key_lens, const int32_t* q_pos,
             float scale, void* workspace, size_t ws_bytes, attn_stream_t stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || S <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !finite_positive(scale)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_F16 && dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hq > 65535 || Hkv > 65535) return ATTN_ERR_UNSUPPORTED;
  if (dtype == ATTN_F32)
    return bwd_f32(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, T, S, D, causal, key_lens,
                   q_pos, scale, workspace, ws_bytes, stream);
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B * Hq > 0x7fffffffll || (T + 127) / 128 > 65535 || (S + 127) / 128 > 65535)
    return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned4(lse) ||
      (key_lens != nullptr && !aligned4(key_lens)) || (q_pos != nullptr && !aligned4(q_pos)))
    return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_bwd_workspace_size(B, Hq, T);
  if (workspace == nullptr || ws_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;
  attn::tcbwd::Params p{};
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.delta = static_cast<float*>(workspace);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.key_lens = key_lens;
  p.q_pos = q_pos;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.T = T;
  p.S = S;
  p.D = D;
  p.causal = causal ? 1 : 0;
  p.n_qtiles = (T + attn::tcbwd::kBM - 1) / attn::tcbwd::kBM;
  p.n_ktiles = (S + attn::tcbwd::kBM - 1) / attn::tcbwd::kBM;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == ATTN_F16)
    return D == 64 ? launch_bwd_tc<64, true>(p, q, k, v, dout, st)
                   : launch_bwd_tc<128, true>(p, q, k, v, dout, st);
  return D == 64 ? launch_bwd_tc<64, false>(p, q, k, v, dout, st)
                 : launch_bwd_tc<128, false>(p, q, k, v, dout, st);
}

size_t attn_decode_workspace_size(int B, int Hq, int S_max, int D) {
  if (B <= 0 || Hq <= 0 || S_max <= 0 || D <= 0) return 0;
  // per (b, h): partial_slots partials of D + 2 floats (O, maximum,
  // denominator); then the split plan: B + 2 int64 (prefix sums, warp count)
  return (size_t)B * Hq * attn::decode::partial_slots(S_max) * ((size_t)D + 2) * sizeof(float) +
         ((size_t)B + 2) * sizeof(long long);
}

}  // extern "C"

namespace {

// Argument and shape checks of a decode step (everything but the workspace),
// shared by attn_decode and attn_decode_noalloc so that both report the same
// status for the same request.
int decode_validate(const void* q, const void* kcache, const void* vcache,
                    const int32_t* kv_lens, const void* o, const float* lse, int B, int Hq,
                    int Hkv, int S_max, int D, int dtype, float scale) {
  if (!q || !kcache || !vcache || !kv_lens || !o) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || S_max <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !finite_positive(scale)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_F16 && dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if (G > 16 || (G & (G - 1)) != 0) return ATTN_ERR_UNSUPPORTED;
  if (B > 65535 || Hkv > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) ||
      !aligned4(kv_lens) || (lse != nullptr && !aligned4(lse)))
    return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// A validated decode step (attn_decode, attn_decode_append): the workspace
// check and the launches.  k_new / v_new non-null: the new token's rows are
// used for and written into row kv_len - 1 by the split kernel.
int decode_run(const void* q, void* kcache, void* vcache, const int32_t* kv_lens, void* o,
               float* lse, int B, int Hq, int Hkv, int S_max, int D, int dtype, float scale,
               void* workspace, size_t ws_bytes, attn_stream_t stream, const void* k_new,
               const void* v_new) {
  const int G = Hq / Hkv;
  const size_t need = attn_decode_workspace_size(B, Hq, S_max, D);
  if (workspace == nullptr || ws_bytes < need || !aligned16(workspace)) return ATTN_ERR_WORKSPACE;

  attn::decode::Params p;
  if (k_new != nullptr) {
    p.k_new = k_new;
    p.v_new = v_new;
    p.kc_w = kcache;
    p.vc_w = vcache;
  }
  p.q = q;
  p.kc = kcache;
  p.vc = vcache;
  p.kv_lens = kv_lens;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.S_max = S_max;
  p.splits = attn::decode::partial_slots(S_max);
  const size_t slots = (size_t)B * Hq * p.splits;
  p.ws_o = static_cast<float*>(workspace);
  p.ws_m = p.ws_o + slots * D;
  p.ws_l = p.ws_m + slots;
  p.plan = reinterpret_cast<long long*>(p.ws_l + slots);  // 8-byte aligned: D + 2 is even
  p.scale_log2 = scale * kLog2e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == ATTN_BF16) {
    return D == 64 ? launch_decode_d<__nv_bfloat16, 64>(p, G, st)
                   : launch_decode_d<__nv_bfloat16, 128>(p, G, st);
  }
  if (dtype == ATTN_F16) {
    return D == 64 ? launch_decode_d<__half, 64>(p, G, st) : launch_decode_d<__half, 128>(p, G, st);
  }
  return D == 64 ? launch_decode_d<float, 64>(p, G, st) : launch_decode_d<float, 128>(p, G, st);
}

}  // namespace

extern "C" {

int attn_decode(const void* q, const void* kcache, const void* vcache, const int32_t* kv_lens,
                void* o, float* lse, int B, int Hq, int Hkv, int S_max, int D, int dtype,
                float scale, void* workspace, size_t ws_bytes, attn_stream_t stream) {
  const int rc = decode_validate(q, kcache, vcache, kv_lens, o, lse, B, Hq, Hkv, S_max, D, dtype,
                                 scale);
  if (rc != ATTN_OK) return rc;
  // the caches are only read on this path
  return decode_run(q, const_cast<void*>(kcache), const_cast<void*>(vcache), kv_lens, o, lse, B,
                    Hq, Hkv, S_max, D, dtype, scale, workspace, ws_bytes, stream, nullptr,
                    nullptr);
}

int attn_decode_append(const void* q, void* kcache, void* vcache, const void* k_new,
                       const void* v_new, const int32_t* kv_lens, void* o, float* lse, int B,
                       int Hq, int Hkv, int S_max, int D, int dtype, float scale, void* workspace,
                       size_t ws_bytes, attn_stream_t stream) {
  const int rc = decode_validate(q, kcache, vcache, kv_lens, o, lse, B, Hq, Hkv, S_max, D, dtype,
                                 scale);
  if (rc != ATTN_OK) return rc;
  if (!k_new || !v_new) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return ATTN_ERR_INVALID_ARG;
  return decode_run(q, kcache, vcache, kv_lens, o, lse, B, Hq, Hkv, S_max, D, dtype, scale,
                    workspace, ws_bytes, stream, k_new, v_new);
}

}  // extern "C"

// ------------------------------------------------ decode without allocation
//
// Scratch for attn_decode_noalloc: a fixed device array defined here, so a
// caller that cannot allocate device memory still gets a decode workspace.
// Host code must not pass `g_noalloc_scratch` itself to a kernel (on the host
// that name is only a stand-in); its device address is looked up once per
// device with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (first call per
// device does the lookup); nullptr on failure.
void* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_ptr[dev] = ptr;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" {

int attn_decode_noalloc(const void* q, const void* kcache, const void* vcache,
                        const int32_t* kv_lens, void* o, float* lse, int B, int Hq, int Hkv,
                        int S_max, int D, int dtype, float scale, attn_stream_t stream) {
  // The same checks as attn_decode first, so that an invalid or unsupported
  // request is reported as such rather than as too large for the scratch.
  const int rc = decode_validate(q, kcache, vcache, kv_lens, o, lse, B, Hq, Hkv, S_max, D, dtype,
                                 scale);
  if (rc != ATTN_OK) return rc;
  const size_t need = attn_decode_workspace_size(B, Hq, S_max, D);
  if (need > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;
  void* scratch = noalloc_scratch();
  if (scratch == nullptr) return ATTN_ERR_CUDA;
  return attn_decode(q, kcache, vcache, kv_lens, o, lse, B, Hq, Hkv, S_max, D, dtype, scale,
                     scratch, ATTN_NOALLOC_SCRATCH_BYTES, stream);
}

int kv_cache_append(void* kcache, void* vcache, const void* k_new, const void* v_new,
                    const int32_t* pos, int B, int Hkv, int S_max, int D, int dtype,
                    int* dev_status, attn_stream_t stream) {
  if (!kcache || !vcache || !k_new || !v_new || !pos) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || Hkv <= 0 || S_max <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  size_t esz;
  if (dtype == ATTN_BF16 || dtype == ATTN_F16) esz = 2;
  else if (dtype == ATTN_F32) esz = 4;
  else return ATTN_ERR_INVALID_ARG;
  const size_t row_bytes = (size_t)D * esz;
  if (row_bytes % 16 != 0) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(kcache) || !aligned16(vcache) || !aligned16(k_new) || !aligned16(v_new) ||
      !aligned4(pos) || (dev_status != nullptr && !aligned4(dev_status)))
    return ATTN_ERR_INVALID_ARG;
  const int vec_per_row = (int)(row_bytes / 16);
  const long long total = (long long)B * Hkv * vec_per_row;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 148 * 16) blocks = 148 * 16;
  attn::kv_append_kernel<<<(unsigned)blocks, threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(kcache), static_cast<uint4*>(vcache), static_cast<const uint4*>(k_new),
      static_cast<const uint4*>(v_new), pos, B, Hkv, S_max, vec_per_row, dev_status);
  return launch_status();
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK: success";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG: invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED: unsupported shape or type";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE: decode workspace missing or too small";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: CUDA error at launch";
    default: return "unknown attn status";
  }
}

unsigned long long attn_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int attn_selftest_wait_timeout(attn_stream_t stream) {
  attn::selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>();
  return launch_status();
}

int attn_device_error(int* code, int clear) {
  int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&v, attn::g_attn_error, sizeof(int)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (code != nullptr) *code = v;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(attn::g_attn_error, &zero, sizeof(int)) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

}  // extern "C"
