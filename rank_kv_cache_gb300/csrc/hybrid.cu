// Decode over a hybrid cache: a dense segment (attention-sink tokens and the recent window, kept
// as a standard KV cache) next to the G-LRD latent middle.
//
// "PuzzleKV" section 3: the sink page and the local window stay dense while the other completed
// pages are factorised; each query attends over dense and factorised pages at once and their
// partial results are merged by online softmax. "Shard" section 7: four fp16 sink tokens and a
// 64-token fp16 window around the compressed middle.
//
// The latent middle is decoded by the regular decode kernels (its output o_mid normalised by its
// own softmax, and its natural-log lse). merge_dense_kernel then takes one CTA per (batch row,
// head): it rotates the query at q_pos (RoPE path; the dense keys are stored rotated at their own
// positions), scores the row's dense tokens (8 warps, each loading four of its tokens at a time
// before scoring them; each lane holds d_h / 32 dimensions, scores reduced across the warp), runs an
// online softmax per warp
// with the p v accumulation, merges the warps, and finally merges the dense segment with the
// middle:
//   lse = ln(e^lse_mid + sum_dense e^s),   out *= e^(lse_mid - lse),   out_dense = sum p v / e^lse
// so that head i's attention output is out_i B_v^(i) + out_dense_i.
#include "internal.h"

namespace palu {
namespace {

constexpr int kHThreads = 256;
constexpr int kHWarps = kHThreads / 32;
constexpr int kHMaxDh = 128;

constexpr int kHAhead = 4;   // tokens each warp loads before scoring them

// `per` (<= 4) consecutive elements at index i as floats; one 8-byte load for four 16-bit values
__device__ __forceinline__ void load_row_part(const void* p, int dtype, int64_t i, int per, float (&x)[4]) {
  if (per == 4 && dtype != kF32) {
    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p) + i);
    const uint32_t w[2] = {u.x, u.y};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (dtype == kF16) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
        x[2 * j] = f.x;
        x[2 * j + 1] = f.y;
      } else {
        x[2 * j] = __uint_as_float(w[j] << 16);
        x[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
      }
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] = e < per ? load_as_f32(p, dtype, i + e) : 0.f;
}

__global__ void __launch_bounds__(kHThreads) merge_dense_kernel(DenseArgs d) {
  __shared__ float qs[kHMaxDh];
  __shared__ float wm[kHWarps], wl[kHWarps];
  __shared__ float wacc[kHWarps][kHMaxDh];
  __shared__ float fin[1], fw[kHWarps];
  const int i = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int dh = d.dh, half = dh / 2, per = dh / 32;
  const int64_t bh = (int64_t)b * d.n_heads + i;

  int D = d.n_tokens[b];
  if (D < 0 || D > d.capacity) {
    if (threadIdx.x == 0 && i == 0) record_error(d.err, kCodeDevice, kErrSeqLen, D, b);
    D = D < 0 ? 0 : int(d.capacity);
  }
  // the query, rotated at q_pos on the RoPE path, pre-scaled by log2(e) / sqrt(d_h)
  const int64_t qoff = bh * dh;
  if (d.rope) {
    int qp = d.q_pos[b];
    if (qp < 0 || qp >= d.max_pos) {
      if (threadIdx.x == 0 && i == 0) record_error(d.err, kCodeDevice, kErrQueryPos, qp, b);
      qp = qp < 0 ? 0 : int(d.max_pos - 1);
    }
    for (int k = threadIdx.x; k < half; k += kHThreads) {
      const float2 cs = d.rope_tab[(int64_t)qp * half + k];
      const float x0 = load_as_f32(d.q, d.q_dtype, qoff + k), x1 = load_as_f32(d.q, d.q_dtype, qoff + k + half);
      qs[k] = (x0 * cs.x - x1 * cs.y) * d.qscale;
      qs[k + half] = (x1 * cs.x + x0 * cs.y) * d.qscale;
    }
  } else {
    for (int k = threadIdx.x; k < dh; k += kHThreads) qs[k] = load_as_f32(d.q, d.q_dtype, qoff + k) * d.qscale;
  }
  __syncthreads();
  float qv[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) qv[e] = e < per ? qs[lane * per + e] : 0.f;

  // online softmax of this warp's tokens (base 2)
  float m = -INFINITY, l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  // warp w takes tokens w, w + 8, ...; each round loads kHAhead tokens' rows before scoring them
  for (int t0 = warp; t0 < D; t0 += kHWarps * kHAhead) {
    float kv[kHAhead][4], vv[kHAhead][4];
#pragma unroll
    for (int a = 0; a < kHAhead; ++a) {
      const int t = t0 + a * kHWarps;
      const int64_t row = (((int64_t)b * d.capacity + (t < D ? t : 0)) * d.n_heads + i) * dh + lane * per;
      load_row_part(d.k, d.dtype, row, per, kv[a]);
      load_row_part(d.v, d.dtype, row, per, vv[a]);
    }
#pragma unroll
    for (int a = 0; a < kHAhead; ++a) {
      if (t0 + a * kHWarps >= D) break;   // warp-uniform
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) s = fmaf(qv[e], kv[a][e], s);
      s = warp_sum(s);
      const float mn = fmaxf(m, s);
      const float al = m == -INFINITY ? 0.f : exp2f(m - mn);
      const float p = exp2f(s - mn);
      l = l * al + p;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] = acc[e] * al + p * vv[a][e];
      m = mn;
    }
  }
  if (lane == 0) {
    wm[warp] = m;
    wl[warp] = l;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (e < per) wacc[warp][lane * per + e] = acc[e];
  __syncthreads();

  // the dense segment's (max, sum) over the warps, then the merge with the middle (natural log):
  // sum_t 2^s_t v_t = sum_w 2^m_w acc_w, so warp w's partial enters out_dense with 2^(m_w) / e^lse
  if (threadIdx.x == 0) {
    constexpr float kLn2 = 0.69314718055994531f;
    float M = -INFINITY;
    for (int w = 0; w < kHWarps; ++w) M = fmaxf(M, wm[w]);
    float L = 0.f;
    for (int w = 0; w < kHWarps; ++w)
      if (wm[w] != -INFINITY) L += wl[w] * exp2f(wm[w] - M);
    const float lse_mid = d.lse[bh];
    const float lse_den = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    const float top = fmaxf(lse_mid, lse_den);
    float lse = -INFINITY;
    if (top != -INFINITY)
      lse = top + logf((lse_mid == -INFINITY ? 0.f : expf(lse_mid - top)) +
                       (lse_den == -INFINITY ? 0.f : expf(lse_den - top)));
    fin[0] = (lse == -INFINITY || lse_mid == -INFINITY) ? 0.f : expf(lse_mid - lse);   // weight of the middle
    for (int w = 0; w < kHWarps; ++w)
      fw[w] = (lse == -INFINITY || wm[w] == -INFINITY) ? 0.f : exp2f(wm[w] - lse / kLn2);
    d.lse[bh] = lse;
  }
  __syncthreads();
  const float w_mid = fin[0];
  for (int c = threadIdx.x; c < d.rv; c += kHThreads) d.out[bh * d.rv + c] *= w_mid;
  for (int c = threadIdx.x; c < dh; c += kHThreads) {
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kHWarps; ++w) o = fmaf(fw[w], wacc[w][c], o);
    d.out_dense[bh * dh + c] = o;
  }
}

}  // namespace

cudaError_t launch_merge_dense(const DenseArgs& d, cudaStream_t st) {
  if (d.batch == 0) return cudaSuccess;
  dim3 grid((unsigned)d.n_heads, (unsigned)d.batch);
  merge_dense_kernel<<<grid, kHThreads, 0, st>>>(d);
  return cudaGetLastError();
}

}  // namespace palu
