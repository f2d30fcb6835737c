// Shared device helpers for the G-LRD decode-attention kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace palu {

enum DType : int { kF32 = 0, kF16 = 1, kBF16 = 2, kINT4 = 3 };
enum Mode : int { kRope = 0, kAbsorbed = 1 };

// Device error word at the start of the workspace. The first recorded error
// wins; later ones are dropped. Codes match palu_status_t.
struct ErrWord {
  unsigned code;
  unsigned where;
  int index;
  int batch;
};
enum ErrWhere : unsigned {
  kErrPosition = 1,   // a token position outside the RoPE table
  kErrSeqLen = 2,     // seq_lens[b] above the launch's max_seq_len / capacity
  kErrSlot = 3,       // an append slot outside the cache
  kErrQueryPos = 4,   // q_pos outside the RoPE table
  kErrWait = 5,       // a bounded mbarrier wait gave up
};
constexpr unsigned kCodeDevice = 4;   // PALU_ERR_DEVICE
constexpr unsigned kCodeTimeout = 5;  // PALU_ERR_TIMEOUT

__device__ __forceinline__ void record_error(ErrWord* e, unsigned code, unsigned where, int index,
                                             int batch) {
  if (atomicCAS(&e->code, 0u, code) == 0u) {
    e->where = where;
    e->index = index;
    e->batch = batch;
  }
}

// ---------------------------------------------------------------------------
// Scalar conversions
// ---------------------------------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ float load_as_f32(const void* p, int dtype, int64_t i) {
  switch (dtype) {
    case kF16: return __half2float(static_cast<const __half*>(p)[i]);
    case kBF16: return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    default: return static_cast<const float*>(p)[i];
  }
}

// Tag type for int4 latents (two signed 4-bit codes per byte + fp16 scale per row).
struct Int4 {};

// Signed code of element e of a packed int4 row: element 2j is the low nibble of
// byte j, element 2j+1 the high nibble, both 4-bit two's complement.
__device__ __forceinline__ int int4_code(const uint8_t* row, int e) {
  const unsigned byte = row[e >> 1];
  const int v = (e & 1) ? int(byte >> 4) : int(byte & 0xFu);
  return (v ^ 8) - 8;
}

// One latent element as fp32. `row` points at the start of the (token, group) row.
template <typename T> struct Latent {
  static __device__ __forceinline__ float get(const void* base, const __half* /*scale*/, int64_t row,
                                              int rank, int e) {
    return to_f32(static_cast<const T*>(base)[row * rank + e]);
  }
  static constexpr int kElemBytesTimes2 = 2 * sizeof(T);
};
template <> struct Latent<Int4> {
  static __device__ __forceinline__ float get(const void* base, const __half* scale, int64_t row,
                                              int rank, int e) {
    const uint8_t* r = static_cast<const uint8_t*>(base) + row * (rank / 2);
    // code * scale is exact in fp32 (4 + 11 significant bits)
    return float(int4_code(r, e)) * __half2float(scale[row]);
  }
  static constexpr int kElemBytesTimes2 = 1;
};

// ---------------------------------------------------------------------------
// Warp reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace palu
