// CUDA-core decode attention over G-LRD latents, both modes, every latent dtype.
//
// One CTA per (split, group, batch row). It streams its T-range of the group's
// latent rows in tiles of kSimtTile tokens, scores them for all s heads of the
// group, keeps an online softmax per head and accumulates p H_v in latent space.
// Output: split partials (m, l, o), merged by the last CTA of each unit (or by the merge
// kernel when the caller provides no counters).
//
// RoPE mode ("Palu" notes, RoPE paragraph and the online-rebuild kernel paragraph):
//   K[t] = H_k[t] B_k,g (all s heads at once), then for head j
//   score = sum_k cos(p w_k) (q_a k_a + q_b k_b) + sin(p w_k) (q_b k_a - q_a k_b)
//   with (a, b) = (k, k + d_h/2), which is q_rot . RoPE(K_j[t], p) written per pair.
// Absorbed mode (key-fusion paragraph): score = q' . H_k[t] with q' = q B_k^T.
// Queries arrive pre-scaled by log2(e)/sqrt(d_h); the softmax works in base 2.
#include "internal.h"
#include "split_merge.cuh"

namespace palu {

namespace {

constexpr int kThreads = 256;
constexpr int kAccMax = 8;   // s * r_v <= 8 * 256

template <int MODE, typename KT, typename VT, typename BT>
__global__ void __launch_bounds__(kThreads) decode_simt_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) float smem[];
  constexpr int TT = kSimtTile;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int s = a.s, dh = a.dh, rk = a.rk, rv = a.rv, half = dh / 2;
  const int qw = (MODE == kRope) ? dh : rk;
  const int cols = s * dh;

  float* q_s = smem;                   // [s][qw]
  float* hk_s = q_s + s * qw;          // [TT][rk]
  float* hv_s = hk_s + TT * rk;        // [TT][rv]
  float* sc_s = hv_s + TT * rv;        // [TT][s] scores, then p
  float* st_s = sc_s + TT * s;         // m[s], l[s], alpha[s]
  float* kr_s = st_s + 3 * 8;          // [TT][cols] rebuilt keys (RoPE mode)

  // sequence length of this row (clamped, errors recorded)
  int T = a.seq_lens[b];
  if (T < 0 || T > a.max_seq_len) {
    if (tid == 0 && split == 0 && g == 0) record_error(a.err, kCodeDevice, kErrSeqLen, T, b);
    T = T < 0 ? 0 : a.max_seq_len;
  }
  const int span = a.tiles_per_split * TT;
  const int t_begin = split * span;
  const int t_end = min(T, t_begin + span);

  for (int i = tid; i < s * qw; i += kThreads) {
    const int j = i / qw, c = i % qw;
    q_s[i] = a.qbuf[((int64_t)b * a.n_heads + g * s + j) * qw + c];
  }
  if (tid < s) {
    st_s[tid] = -INFINITY;  // m
    st_s[8 + tid] = 0.f;    // l
  }
  float acc[kAccMax];
#pragma unroll
  for (int k = 0; k < kAccMax; ++k) acc[k] = 0.f;

  // the cache group this kernel group reads (split groups share their cache group's latents)
  const int gs = a.g_split > 1 ? a.g_split : 1;
  const int cache_g = g / gs, cache_n_g = a.n_g / gs;
  for (int t0 = t_begin; t0 < t_end; t0 += TT) {
    const int nt = min(TT, t_end - t0);
    __syncthreads();
    for (int i = tid; i < TT * rk; i += kThreads) {
      const int t = i / rk, c = i % rk;
      const int64_t row = ((int64_t)b * a.capacity + (t0 + t)) * cache_n_g + cache_g;
      hk_s[i] = (t < nt) ? Latent<KT>::get(a.hk, a.k_scale, row, rk, c) : 0.f;
    }
    for (int i = tid; i < TT * rv; i += kThreads) {
      const int t = i / rv, c = i % rv;
      const int64_t row = ((int64_t)b * a.capacity + (t0 + t)) * cache_n_g + cache_g;
      hv_s[i] = (t < nt) ? Latent<VT>::get(a.hv, a.v_scale, row, rv, c) : 0.f;
    }
    __syncthreads();

    if (MODE == kRope) {
      // rebuild K[t][col] = sum_m H_k[t][m] B_k[g][m][col] for the whole tile
      const BT* bkg = static_cast<const BT*>(a.bk) + (int64_t)g * rk * cols;
      for (int col = tid; col < cols; col += kThreads) {
        float kt[TT];
#pragma unroll
        for (int t = 0; t < TT; ++t) kt[t] = 0.f;
        for (int m = 0; m < rk; ++m) {
          const float bv = to_f32(bkg[(int64_t)m * cols + col]);
#pragma unroll
          for (int t = 0; t < TT; ++t) kt[t] = fmaf(hk_s[t * rk + m], bv, kt[t]);
        }
#pragma unroll
        for (int t = 0; t < TT; ++t) kr_s[t * cols + col] = kt[t];
      }
      __syncthreads();
      // scores: 4 threads per (token, head) pair, each over a quarter of the pairs
      for (int base = 0; base < TT * s * 4; base += kThreads) {
        const int idx = base + tid;
        const int pr = idx >> 2, part = idx & 3;
        float sc = 0.f;
        int t = 0, j = 0;
        if (pr < TT * s) {
          t = pr / s;
          j = pr % s;
          if (t < nt) {
            int pos = t0 + t;
            if (a.positions) pos = a.positions[(int64_t)b * a.capacity + t0 + t];
            if (pos < 0 || pos >= a.max_pos) {
              if (part == 0) record_error(a.err, kCodeDevice, kErrPosition, pos, b);
              pos = pos < 0 ? 0 : int(a.max_pos - 1);
            }
            const float2* cs = a.rope + (int64_t)pos * half;
            const float* kj = kr_s + t * cols + j * dh;
            const float* qj = q_s + j * dh;
            for (int k = part; k < half; k += 4) {
              const float ka = kj[k], kb = kj[k + half];
              const float qa = qj[k], qb = qj[k + half];
              const float2 c = cs[k];
              sc = fmaf(c.x, fmaf(qa, ka, qb * kb), sc);
              sc = fmaf(c.y, fmaf(qb, ka, -qa * kb), sc);
            }
          }
        }
        sc += __shfl_xor_sync(0xffffffffu, sc, 1);
        sc += __shfl_xor_sync(0xffffffffu, sc, 2);
        if (pr < TT * s && part == 0) sc_s[t * s + j] = (t < nt) ? sc : -INFINITY;
      }
    } else {
      for (int base = 0; base < TT * s * 4; base += kThreads) {
        const int idx = base + tid;
        const int pr = idx >> 2, part = idx & 3;
        float sc = 0.f;
        int t = 0, j = 0;
        if (pr < TT * s) {
          t = pr / s;
          j = pr % s;
          if (t < nt) {
            const float* h = hk_s + t * rk;
            const float* qj = q_s + j * rk;
            for (int m = part; m < rk; m += 4) sc = fmaf(qj[m], h[m], sc);
          }
        }
        sc += __shfl_xor_sync(0xffffffffu, sc, 1);
        sc += __shfl_xor_sync(0xffffffffu, sc, 2);
        if (a.alibi && pr < TT * s && t < nt) {
          // ALiBi: m_i (pos_t - q_pos) log2(e), m_i = 2^(-8 (i + 1) / n) for head i = g s + j
          const int pos = a.positions ? a.positions[(int64_t)b * a.capacity + t0 + t] : t0 + t;
          int qp = a.positions ? a.positions[(int64_t)b * a.capacity + T - 1] : T - 1;
          if (a.q_pos) qp = a.q_pos[b];
          const float m = exp2f(-8.f * float(g * s + j + 1) / float(a.n_heads)) * 1.4426950408889634f;
          sc = fmaf(m, float(pos) - float(qp), sc);
        }
        if (pr < TT * s && part == 0) sc_s[t * s + j] = (t < nt) ? sc : -INFINITY;
      }
    }
    __syncthreads();

    // online softmax update, one thread per head
    if (tid < s) {
      const int j = tid;
      const float m_old = st_s[j];
      float mx = m_old;
      for (int t = 0; t < TT; ++t) mx = fmaxf(mx, sc_s[t * s + j]);
      const bool none = (mx == -INFINITY);
      const float alpha = none ? 1.f : exp2f(m_old - mx);
      float lsum = 0.f;
      for (int t = 0; t < TT; ++t) {
        const float p = none ? 0.f : exp2f(sc_s[t * s + j] - mx);
        sc_s[t * s + j] = p;
        lsum += p;
      }
      st_s[j] = mx;
      st_s[8 + j] = st_s[8 + j] * alpha + lsum;
      st_s[16 + j] = alpha;
    }
    __syncthreads();

    // o[j][c] = alpha_j o[j][c] + sum_t p[t][j] H_v[t][c]
#pragma unroll
    for (int k = 0; k < kAccMax; ++k) {
      const int idx = tid + k * kThreads;
      if (idx < s * rv) {
        const int j = idx / rv, c = idx % rv;
        float o = acc[k] * st_s[16 + j];
        for (int t = 0; t < nt; ++t) o = fmaf(sc_s[t * s + j], hv_s[t * rv + c], o);
        acc[k] = o;
      }
    }
  }

  // split partials
#pragma unroll
  for (int k = 0; k < kAccMax; ++k) {
    const int idx = tid + k * kThreads;
    if (idx < s * rv) {
      const int j = idx / rv, c = idx % rv;
      const int64_t bh = (int64_t)b * a.n_heads + g * s + j;
      a.part_o[(bh * a.n_splits + split) * rv + c] = acc[k];
    }
  }
  __syncthreads();
  if (tid < s) {
    const int64_t bh = (int64_t)b * a.n_heads + g * s + tid;
    a.part_ml[bh * a.n_splits + split] = make_float2(st_s[tid], st_s[8 + tid]);
  }
  __shared__ int merge_flag;
  __syncthreads();  // the tile buffers are free: reuse them as merge scratch (s * (n_splits + 2) floats)
  merge_if_last(a, b, g * s, s, &merge_flag, hk_s);
}

size_t simt_smem_bytes(int mode, const DecodeArgs& a) {
  const int TT = kSimtTile;
  const int qw = (mode == kRope) ? a.dh : a.rk;
  size_t f = (size_t)a.s * qw + (size_t)TT * a.rk + (size_t)TT * a.rv + (size_t)TT * a.s + 24;
  if (mode == kRope) f += (size_t)TT * a.s * a.dh;
  // the split merge reuses everything after the query block as scratch
  const size_t merge = (size_t)a.s * qw + (size_t)a.s * (a.n_splits + 2) + 16;
  return (f > merge ? f : merge) * sizeof(float);
}

template <int MODE, typename KT, typename VT, typename BT>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t st) {
  const size_t smem = simt_smem_bytes(MODE, a);
  auto kern = decode_simt_kernel<MODE, KT, VT, BT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_splits, a.n_g, a.batch);
  kern<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_mode(const DecodeArgs& a, cudaStream_t st) {
  if (a.k_dtype == kF32) return launch_t<MODE, float, float, float>(a, st);
  if (a.k_dtype == kF16)
    return a.v_dtype == kINT4 ? launch_t<MODE, __half, Int4, __half>(a, st) : launch_t<MODE, __half, __half, __half>(a, st);
  if (a.k_dtype == kBF16)
    return a.v_dtype == kINT4 ? launch_t<MODE, __nv_bfloat16, Int4, __nv_bfloat16>(a, st)
                              : launch_t<MODE, __nv_bfloat16, __nv_bfloat16, __nv_bfloat16>(a, st);
  return launch_t<MODE, Int4, Int4, __half>(a, st);
}

}  // namespace

cudaError_t launch_decode_simt(int mode, const DecodeArgs& a, cudaStream_t st) {
  if (a.s * a.rv > kAccMax * kThreads || a.s > 8) return cudaErrorInvalidValue;
  return mode == kRope ? launch_mode<kRope>(a, st) : launch_mode<kAbsorbed>(a, st);
}

}  // namespace palu
