// Set-up and small per-call kernels: RoPE table, B_k copies, query preparation,
// split-T merge, latent append/quantisation and the int4 debug export.
#include <math.h>

#include "internal.h"

namespace palu {

// ---------------------------------------------------------------------------
// RoPE table: tab[p][k] = (cos(p w_k), sin(p w_k)), w_k = theta^(-2k/d_h), computed in
// float64 and rounded to float32 once (rotate-half RoPE with the RoFormer schedule).
// ---------------------------------------------------------------------------
// Also phase[k] = frac(w_k / 2pi) as a 64-bit fixed-point fraction of a turn, so that the
// phase of position p is the top bits of p * phase[k] mod 2^64 (phase accumulation as in
// direct digital synthesis): exact integer range reduction for every position.
__global__ void rope_table_kernel(float2* tab, uint64_t* phase, int64_t max_pos, int half, int dh, double theta) {
  const int64_t n = max_pos * half;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = i / half;
    const int k = int(i % half);
    const double w = pow(theta, -2.0 * double(k) / double(dh));
    double sn, cs;
    sincos(double(p) * w, &sn, &cs);
    tab[i] = make_float2(float(cs), float(sn));
    if (p == 0) {
      const double turns = w / 6.283185307179586476925286766559;
      const double v = ldexp(turns - floor(turns), 64);
      phase[k] = v >= 18446744073709549568.0 ? ~0ull : __double2ull_rn(v);
    }
  }
}

cudaError_t launch_rope_table(float2* tab, uint64_t* phase, int64_t max_pos, int dh, double theta, cudaStream_t st) {
  const int64_t n = max_pos * (dh / 2);
  const int blocks = int((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  rope_table_kernel<<<blocks, 256, 0, st>>>(tab, phase, max_pos, dh / 2, dh, theta);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// B_k copies: dst = B_k as given ([n_g][rk][cols]); dst_t = its per-group transpose
// [n_g][cols][rk] in the MMA operand type (the K-major B operand of the rebuild GEMM).
// ---------------------------------------------------------------------------
// dst_t = B_k^T as the tensor-core kernel's K-major operand, [n_g][s * d_h][r]. With an even
// group size the rows of each head pair are interleaved by head (row 2 d + (j & 1) of pair j / 2
// holds dimension d of head j), so the MMA writes the two heads' values of a dimension into
// adjacent accumulator columns and the epilogue updates both heads with one packed instruction.
// perm8 (int4 caches): within each group of eight ranks, position p holds rank [0,2,4,6,1,3,5,7][p],
// the order in which the int4 converter emits a packed word's codes; permuting K in both MMA
// operands alike leaves the product unchanged.
// pack > 1 (packed groups, 16-bit B_k only): the n_g x rk x cols copy is the block-diagonal B_k of
// kernel groups made of `pack` source groups of src_s heads and src_rk ranks: source group jg of
// kernel group g fills ranks [jg src_rk, (jg + 1) src_rk) x its own heads' columns, zeros elsewhere.
// split > 1 (split groups): kernel group g is column block g % split (cols wide) of source group
// g / split, whose rows hold src_s * dh columns.
__global__ void copy_bk_kernel(const void* src, int bk_dtype, void* dst, void* dst_t, int mma_dtype, int n_g,
                               int rk, int cols, int dh, int perm8, int pack, int split, int src_s, int src_rk) {
  const int64_t n = (int64_t)n_g * rk * cols;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int c = int(i % cols);
    const int m = int((i / cols) % rk);
    const int g = int(i / ((int64_t)cols * rk));
    const int esz = bk_dtype == kF32 ? 4 : 2;
    // the source element: the same index, or for packed groups the block-diagonal expansion
    int64_t si = i;
    if (split > 1) si = ((int64_t)(g / split) * rk + m) * ((int64_t)src_s * dh) + (int64_t)(g % split) * cols + c;
    if (pack > 1) {
      const int jg = (c / dh) / src_s;   // source group of this column within the kernel group
      si = (m / src_rk == jg) ? (((int64_t)g * pack + jg) * src_rk + (m - jg * src_rk)) * ((int64_t)src_s * dh) +
                                    (c - jg * src_s * dh)
                              : -1;
    }
    // plain byte copy of the original layout
    if (esz == 4) static_cast<float*>(dst)[i] = si >= 0 ? static_cast<const float*>(src)[si] : 0.f;
    else static_cast<uint16_t*>(dst)[i] = si >= 0 ? static_cast<const uint16_t*>(src)[si] : uint16_t(0);
    if (dst_t) {
      const float v = si >= 0 ? load_as_f32(src, bk_dtype, si) : 0.f;
      const int j = c / dh, d = c % dh;
      const int ct = ((cols / dh) % 2 == 0) ? (j / 2) * 2 * dh + 2 * d + (j & 1) : c;
      const int mt = perm8 ? (m & ~7) | ((m & 1) << 2) | ((m & 7) >> 1) : m;
      const int64_t o = ((int64_t)g * cols + ct) * rk + mt;
      if (mma_dtype == kBF16) static_cast<__nv_bfloat16*>(dst_t)[o] = __float2bfloat16_rn(v);
      else static_cast<__half*>(dst_t)[o] = __float2half_rn(v);
    }
  }
}

cudaError_t launch_copy_bk(const void* src, int bk_dtype, void* dst, void* dst_t, int mma_dtype, int n_g, int rk,
                           int cols, int dh, int perm8, int pack, int split, int src_s, int src_rk, cudaStream_t st) {
  const int64_t n = (int64_t)n_g * rk * cols;
  const int blocks = int((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  copy_bk_kernel<<<blocks, 256, 0, st>>>(src, bk_dtype, dst, dst_t, mma_dtype, n_g, rk, cols, dh, perm8, pack, split,
                                         src_s, src_rk);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Shared helpers for sequence length and positions
// ---------------------------------------------------------------------------
__device__ __forceinline__ int clamp_seq_len(const DecodeArgs& a, int b) {
  int T = a.seq_lens[b];
  const int lim = a.max_seq_len;
  if (T < 0 || T > lim) {
    record_error(a.err, kCodeDevice, kErrSeqLen, T, b);
    T = T < 0 ? 0 : lim;
  }
  return T;
}

// ---------------------------------------------------------------------------
// Query preparation (one block per (b, head)):
//   RoPE mode:     q_rot = RoPE(q, q_pos) * qscale                       -> [B][n][dh]
//   absorbed mode: q'    = (B_k[g][:, j block] q) * qscale  (q B_k^T)    -> [B][n][rk]
// qscale = log2(e)/sqrt(d_h), so the decode kernels take exp2 of the scores.
// ---------------------------------------------------------------------------
__global__ void qprep_rope_kernel(const void* q, int q_dtype, DecodeArgs a, const int32_t* q_pos, float qscale,
                                  float* qbuf) {
  const int b = blockIdx.x / a.n_heads;
  const int i = blockIdx.x % a.n_heads;
  const int half = a.dh / 2;
  const int T = clamp_seq_len(a, b);
  int qp = 0;
  if (q_pos) qp = q_pos[b];
  else if (T > 0) qp = a.positions ? a.positions[(int64_t)b * a.capacity + (T - 1)] : (T - 1);
  if (qp < 0 || qp >= a.max_pos) {
    if (threadIdx.x == 0) record_error(a.err, kCodeDevice, kErrQueryPos, qp, b);
    qp = qp < 0 ? 0 : int(a.max_pos - 1);
  }
  const int64_t qoff = ((int64_t)b * a.n_heads + i) * a.dh;
  for (int k = threadIdx.x; k < half; k += blockDim.x) {
    const float2 cs = a.rope[(int64_t)qp * half + k];
    const float x0 = load_as_f32(q, q_dtype, qoff + k);
    const float x1 = load_as_f32(q, q_dtype, qoff + k + half);
    qbuf[qoff + k] = (x0 * cs.x - x1 * cs.y) * qscale;
    qbuf[qoff + k + half] = (x1 * cs.x + x0 * cs.y) * qscale;
  }
}

__global__ void qprep_absorbed_kernel(const void* q, int q_dtype, DecodeArgs a, float qscale, float* qbuf) {
  extern __shared__ float qs[];
  const int b = blockIdx.x / a.n_heads;
  const int i = blockIdx.x % a.n_heads;
  const int g = i / a.s, j = i % a.s;
  const int cols = a.s * a.dh;
  const int64_t qoff = ((int64_t)b * a.n_heads + i) * a.dh;
  for (int c = threadIdx.x; c < a.dh; c += blockDim.x) qs[c] = load_as_f32(q, q_dtype, qoff + c);
  __syncthreads();
  for (int m = threadIdx.x; m < a.rk; m += blockDim.x) {
    const int64_t row = ((int64_t)g * a.rk + m) * cols + (int64_t)j * a.dh;
    float acc = 0.f;
    for (int c = 0; c < a.dh; ++c) acc = fmaf(load_as_f32(a.bk, a.bk_dtype, row + c), qs[c], acc);
    qbuf[((int64_t)b * a.n_heads + i) * a.rk + m] = acc * qscale;
  }
}

cudaError_t launch_qprep(int mode, const void* q, int q_dtype, const DecodeArgs& a, const int32_t* q_pos,
                         float qscale, float* qbuf, cudaStream_t st) {
  const int blocks = a.batch * a.n_heads;
  if (mode == kRope) qprep_rope_kernel<<<blocks, 64, 0, st>>>(q, q_dtype, a, q_pos, qscale, qbuf);
  else qprep_absorbed_kernel<<<blocks, 256, a.dh * sizeof(float), st>>>(q, q_dtype, a, qscale, qbuf);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Split-T merge (flash-decoding): with partials (m_k, l_k, o_k) in log2 units,
//   M = max m_k, L = sum l_k 2^(m_k - M), o = sum o_k 2^(m_k - M) / L, lse = ln2 (M + log2 L).
// One block per (b, head); empty rows give o = 0, lse = -inf.
// ---------------------------------------------------------------------------
__global__ void combine_kernel(DecodeArgs a, float* out, float* lse) {
  extern __shared__ float wsh[];  // [n_splits] weights
  const int bh = blockIdx.x;
  const float2* ml = a.part_ml + (int64_t)bh * a.n_splits;
  __shared__ float sM, sInvL, sL;
  if (threadIdx.x < 32) {
    float M = -INFINITY;
    for (int k = threadIdx.x; k < a.n_splits; k += 32) M = fmaxf(M, ml[k].x);
    M = warp_max(M);
    float L = 0.f;
    for (int k = threadIdx.x; k < a.n_splits; k += 32) {
      const float2 v = ml[k];
      const float w = (v.x == -INFINITY) ? 0.f : exp2f(v.x - M);
      wsh[k] = w;
      L += v.y * w;
    }
    L = warp_sum(L);
    if (threadIdx.x == 0) {
      sM = M;
      sL = L;
      sInvL = (L > 0.f) ? 1.f / L : 0.f;
    }
  }
  __syncthreads();
  const float inv = sInvL;
  for (int c = threadIdx.x; c < a.rv; c += blockDim.x) {
    float acc = 0.f;
    const float* po = a.part_o + (int64_t)bh * a.n_splits * a.rv + c;
    for (int k = 0; k < a.n_splits; ++k) {
      const float w = wsh[k];
      if (w != 0.f) acc = fmaf(po[(int64_t)k * a.rv], w, acc);
    }
    out[(int64_t)bh * a.rv + c] = acc * inv;
  }
  if (lse && threadIdx.x == 0) lse[bh] = (sL > 0.f) ? (sM + log2f(sL)) * 0.69314718055994531f : -INFINITY;
}

cudaError_t launch_combine(const DecodeArgs& a, float* out, float* lse, cudaStream_t st) {
  combine_kernel<<<a.batch * a.n_heads, 256, a.n_splits * sizeof(float), st>>>(a, out, lse);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Append: one warp per (b, new token, group) row.
// int4 rows: amax over the row in fp32; scale = fp16_rn(min(amax / 7, 65504)) (IEEE division);
// code = clamp(rint_half_even(h / scale), -7, 7), 0 when the scale is 0; element 2j in the low
// nibble of byte j, 2j+1 in the high nibble.
// ---------------------------------------------------------------------------
struct AppendSide {
  void* cache;
  __half* scale;
  const void* src;
  int rank;
  int dtype;   // this side's cache dtype (values may be int4 while keys are not)
};

__device__ void append_row(const AppendSide& sd, int64_t capacity, int n_g, int src_dtype, const int32_t* dst_slot,
                           int n_new, int64_t row, int lane, ErrWord* err) {
  const int rank = sd.rank;
  const int cache_dtype = sd.dtype;
  const int g = int(row % n_g);
  const int i = int((row / n_g) % n_new);
  const int b = int(row / ((int64_t)n_g * n_new));
  const int dst = dst_slot[b] + i;
  if (dst < 0 || dst >= capacity) {
    if (lane == 0) record_error(err, kCodeDevice, kErrSlot, dst, b);
    return;
  }
  const int64_t src_off = row * rank;
  const int64_t crow = ((int64_t)b * capacity + dst) * n_g + g;
  // each lane owns `per` consecutive elements (rank / 32 = 2, 4 or 8); every load is issued
  // before the first store, so a row costs one memory latency
  const int per = rank / 32;
  float h[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (k < per) h[k] = load_as_f32(sd.src, src_dtype, src_off + lane * per + k);
  if (cache_dtype != kINT4) {
    const int64_t o = crow * rank + lane * per;
    if (cache_dtype == kF32) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < per) static_cast<float*>(sd.cache)[o + k] = h[k];
    } else if (per == 8) {
      // one 16-byte store of eight 16-bit values (rows are 16-byte aligned)
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (cache_dtype == kF16) {
          const __half2 v = __floats2half2_rn(h[2 * j], h[2 * j + 1]);
          w[j] = *reinterpret_cast<const uint32_t*>(&v);
        } else {
          const __nv_bfloat162 v = __floats2bfloat162_rn(h[2 * j], h[2 * j + 1]);
          w[j] = *reinterpret_cast<const uint32_t*>(&v);
        }
      }
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(sd.cache) + o) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k < per) {
          if (cache_dtype == kF16) static_cast<__half*>(sd.cache)[o + k] = __float2half_rn(h[k]);
          else static_cast<__nv_bfloat16*>(sd.cache)[o + k] = __float2bfloat16_rn(h[k]);
        }
      }
    }
    return;
  }
  // int4: quantise the row with one scale
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (k < per) amax = fmaxf(amax, fabsf(h[k]));
  amax = warp_max(amax);
  const __half sc = __float2half_rn(fminf(__fdiv_rn(amax, 7.0f), 65504.0f));
  const float sf = __half2float(sc);
  uint8_t* out = static_cast<uint8_t*>(sd.cache) + crow * (rank / 2) + lane * (per / 2);
  uint32_t packed = 0;   // byte j = elements 2j (low nibble) and 2j + 1 (high nibble)
#pragma unroll
  for (int k = 0; k < 8; k += 2) {
    if (k < per) {
      int c0 = 0, c1 = 0;
      if (sf != 0.f) {
        c0 = int(fminf(fmaxf(rintf(__fdiv_rn(h[k], sf)), -7.f), 7.f));
        c1 = int(fminf(fmaxf(rintf(__fdiv_rn(h[k + 1], sf)), -7.f), 7.f));
      }
      packed |= uint32_t((c0 & 0xF) | ((c1 & 0xF) << 4)) << (4 * k);
    }
  }
  if (per == 8) {
    *reinterpret_cast<uint32_t*>(out) = packed;   // 4-byte aligned: rows are 128-byte multiples
  } else {
    for (int j = 0; j < per / 2; ++j) out[j] = uint8_t(packed >> (8 * j));
  }
  if (lane == 0) sd.scale[crow] = sc;
}

// One warp per (side, b, new token, group) row; rows of the key cache come first, then the
// value cache, so both are written by one launch.
__global__ void append_kernel(AppendSide k_side, AppendSide v_side, int64_t capacity, int n_g, int src_dtype,
                              const int32_t* dst_slot, int batch, int n_new, ErrWord* err) {
  const int warps = blockDim.x / 32;
  const int64_t gw = (int64_t)blockIdx.x * warps + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)batch * n_new * n_g;
  if (gw >= 2 * rows) return;
  if (gw < rows) append_row(k_side, capacity, n_g, src_dtype, dst_slot, n_new, gw, lane, err);
  else append_row(v_side, capacity, n_g, src_dtype, dst_slot, n_new, gw - rows, lane, err);
}

cudaError_t launch_append(void* cache_k, __half* scale_k, int rank_k, const void* src_k, void* cache_v,
                          __half* scale_v, int rank_v, const void* src_v, int k_dtype, int v_dtype, int64_t capacity,
                          int n_g, int src_dtype, const int32_t* dst_slot, int batch, int n_new, ErrWord* err,
                          cudaStream_t st) {
  const int64_t rows = (int64_t)batch * n_new * n_g;
  if (rows == 0) return cudaSuccess;
  const int warps = 8;
  const int64_t blocks = (2 * rows + warps - 1) / warps;
  append_kernel<<<(unsigned)blocks, warps * 32, 0, st>>>(AppendSide{cache_k, scale_k, src_k, rank_k, k_dtype},
                                                          AppendSide{cache_v, scale_v, src_v, rank_v, v_dtype},
                                                          capacity, n_g, src_dtype, dst_slot, batch, n_new, err);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Debug export of dequantised int4 latents through the CUDA-core decode kernel's unpack routine
// (Latent<Int4>::get); the tensor-core kernel's routines have their own exports in decode_tc.cu.
// ---------------------------------------------------------------------------
__global__ void debug_dequant_kernel(const void* cache, const __half* scale, int64_t capacity, int n_g, int rank,
                                     int batch, int64_t n_tokens, float* out) {
  const int64_t n = (int64_t)batch * n_tokens * n_g * rank;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int e = int(i % rank);
    const int64_t r = i / rank;  // (b, t, g) in the output
    const int g = int(r % n_g);
    const int64_t t = (r / n_g) % n_tokens;
    const int64_t b = r / ((int64_t)n_g * n_tokens);
    const int64_t crow = (b * capacity + t) * n_g + g;
    out[i] = Latent<Int4>::get(cache, scale, crow, rank, e);
  }
}

cudaError_t launch_debug_dequant(const void* cache, const __half* scale, int cache_dtype, int64_t capacity,
                                 int n_g, int rank, int batch, int64_t n_tokens, float* out, cudaStream_t st) {
  if (cache_dtype != kINT4) return cudaErrorInvalidValue;
  const int64_t n = (int64_t)batch * n_tokens * n_g * rank;
  if (n == 0) return cudaSuccess;
  const int blocks = int((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  debug_dequant_kernel<<<blocks, 256, 0, st>>>(cache, scale, capacity, n_g, rank, batch, n_tokens, out);
  return cudaGetLastError();
}

}  // namespace palu
