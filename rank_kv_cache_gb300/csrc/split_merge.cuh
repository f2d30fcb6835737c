// Split-T merge inside the decode kernels (flash-decoding): the last CTA of a unit merges.
#pragma once

#include "internal.h"

namespace palu {

// Log-sum-exp merge of the n_splits partials of heads [h0, h0 + nh) of batch row b, with
// partials (m_k, l_k, o_k) in log2 units: M = max m_k, L = sum l_k 2^(m_k - M),
// o = sum o_k 2^(m_k - M) / L, lse = ln2 (M + log2 L); an empty row gives o = 0, lse = -inf.
// Executed by every thread of the merging CTA. `w` is shared scratch of nh * (n_splits + 2)
// floats: warp j computes head j's weights 2^(m_k - M) and (M, L) once, then all threads form
// the outputs with independent, unrolled loads. Partials written by other CTAs are read
// around L1 (ld.global.cg).
__device__ __forceinline__ void merge_partials(const DecodeArgs& a, int b, int h0, int nh, float* w) {
  const int tid = threadIdx.x, nthreads = blockDim.x, warp = tid >> 5, lane = tid & 31;
  const int ns = a.n_splits;
  float* ML = w + nh * ns;   // [nh][2]: M, L
  if (warp < nh) {
    const int64_t bh = (int64_t)b * a.n_heads + h0 + warp;
    const float2* ml = a.part_ml + bh * ns;
    float M = -INFINITY;
    for (int k = lane; k < ns; k += 32) M = fmaxf(M, __ldcg(&ml[k].x));
    M = warp_max(M);
    float L = 0.f;
    for (int k = lane; k < ns; k += 32) {
      const float2 v = __ldcg(&ml[k]);
      const float wk = (v.x == -INFINITY) ? 0.f : exp2f(v.x - M);
      w[warp * ns + k] = wk;
      L = fmaf(v.y, wk, L);
    }
    L = warp_sum(L);
    if (lane == 0) {
      ML[2 * warp] = M;
      ML[2 * warp + 1] = L;
    }
  }
  __syncthreads();
  // packed groups: head h's output is its own source group's out_rv columns of the rv computed
  const int orv = a.out_rv > 0 ? a.out_rv : a.rv;
  for (int idx = tid; idx < nh * orv; idx += nthreads) {
    const int j = idx / orv, c = idx % orv;
    const int64_t bh = (int64_t)b * a.n_heads + h0 + j;
    const int c0 = a.out_rv > 0 ? (((h0 + j) & 3) / a.pack_s) * orv : 0;
    const float* po = a.part_o + bh * ns * a.rv + c0 + c;
    const float* wj = w + j * ns;
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
    int k = 0;
    for (; k + 4 <= ns; k += 4) {
      const float x0 = __ldcg(po + (int64_t)(k + 0) * a.rv), x1 = __ldcg(po + (int64_t)(k + 1) * a.rv);
      const float x2 = __ldcg(po + (int64_t)(k + 2) * a.rv), x3 = __ldcg(po + (int64_t)(k + 3) * a.rv);
      o0 = fmaf(x0, wj[k + 0], o0);
      o1 = fmaf(x1, wj[k + 1], o1);
      o2 = fmaf(x2, wj[k + 2], o2);
      o3 = fmaf(x3, wj[k + 3], o3);
    }
    for (; k < ns; ++k) o0 = fmaf(__ldcg(po + (int64_t)k * a.rv), wj[k], o0);
    const float o = (o0 + o1) + (o2 + o3);
    const float L = ML[2 * j + 1];
    a.out[bh * orv + c] = L > 0.f ? o / L : 0.f;
    if (a.lse && c == 0) a.lse[bh] = L > 0.f ? (ML[2 * j] + log2f(L)) * 0.69314718055994531f : -INFINITY;
  }
}

// Call from every thread of the CTA after the CTA's partials for heads [h0, h0 + nh) of row b
// are written. `flag` is one shared word, `scratch` shared memory of nh * (n_splits + 2)
// floats that is free at this point. Every CTA counts itself, also after a timed-out wait,
// so the counter always completes and resets.
__device__ __forceinline__ void merge_if_last(const DecodeArgs& a, int b, int h0, int nh, volatile int* flag,
                                              float* scratch) {
  if (!a.counters) return;
  __threadfence();
  __syncthreads();
  unsigned* ctr = a.counters + (int64_t)b * a.n_heads + h0;
  if (threadIdx.x == 0) *flag = (atomicAdd(ctr, 1u) == unsigned(a.n_splits - 1)) ? 1 : 0;
  __syncthreads();
  if (*flag) {
    __threadfence();
    merge_partials(a, b, h0, nh, scratch);
    if (threadIdx.x == 0) *ctr = 0u;
  }
}

}  // namespace palu
