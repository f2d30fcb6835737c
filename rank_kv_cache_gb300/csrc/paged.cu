// Decode over a page-factorised KV cache, next to the dense sink and window tokens.
//
// "PuzzleKV: page-based low-rank decomposition for KV cache compression", section 3.3 (step 4):
// every completed page p of a head holds K_p ~= L_p^K R_p^K and V_p ~= L_p^V R_p^V (L: P x r,
// R: r x d). The page's scores are s_p = (q R_p^K^T) L_p^K^T / sqrt(d) and its values are read as
// p L_p^V R_p^V, without rebuilding the page; dense and factorised pages share one softmax.
//
// One CTA per (split, head, batch row). Warp 0 streams the split's page records (L_K, R_K, L_V,
// R_V of one page and head, contiguous: 640 r bytes in 16-bit storage) with cp.async.bulk into a
// ring of shared-memory slots. Eight consumer warps take the pages round-robin, one page per warp
// at a time; lane t owns token t of the page (P = 32) and head dimensions 4t .. 4t + 3:
//   u = R_K q        per-lane partial dot products, summed over the lanes by a transpose-reduce
//                    that leaves u_j in lane j << (5 - log2 r)
//   s_t = L_K[t] u   the lane's own token (q arrives rotated and scaled by log2(e)/sqrt(d))
//   online softmax in base 2 over the warp's pages
//   w = p L_V        per-lane products p_t L_V[t], transpose-reduced like u
//   o = o alpha + w R_V   the lane's four dimensions
// The warps' states merge in shared memory, the split writes its partial (m, l, o), and the last
// CTA of (batch row, head) merges the splits with the decode kernels' merge. Every mbarrier wait
// is bounded; a wait that gives up records PALU_ERR_TIMEOUT and the CTA drains its copies.
#include "internal.h"
#include "split_merge.cuh"
#include "tc_ptx.cuh"

namespace palu {
namespace {

constexpr int kPgP = 32;                      // tokens per page: one per lane
constexpr int kPgDh = 128;                    // head dimension: four per lane
constexpr int kPgWarps = 8;                   // consumer warps
constexpr int kPgThreads = 32 * (kPgWarps + 1);

template <int R>
struct PgLay {
  static constexpr int kLK = 0;                          // [P][R]
  static constexpr int kRK = kLK + kPgP * R * 2;         // [R][d]
  static constexpr int kLV = kRK + R * kPgDh * 2;        // [P][R]
  static constexpr int kRV = kLV + kPgP * R * 2;         // [R][d]
  static constexpr int kRec = kRV + R * kPgDh * 2;       // 640 R bytes
  // at least one slot per consumer warp; about 80 KB, so two CTAs share an SM for r <= 16
  static constexpr int kSlotsWant = (80 * 1024 / kRec) / kPgWarps * kPgWarps;
  static constexpr int kSlots = kSlotsWant < kPgWarps ? kPgWarps : kSlotsWant;
  static constexpr int kOffBar = kSlots * kRec;
  static constexpr int kOffMisc = kOffBar + 2 * kSlots * 8;       // abort flag, merge flag
  static constexpr int kOffQ = kOffMisc + 16;                     // float [d]
  static constexpr int kOffWm = kOffQ + kPgDh * 4;                // float [warps]
  static constexpr int kOffWl = kOffWm + kPgWarps * 4;            // float [warps]
  static constexpr int kOffWo = kOffWl + kPgWarps * 4;            // float [warps][d]
  static constexpr int kSmem = kOffWo + kPgWarps * kPgDh * 4;
  static_assert(kRec % 16 == 0, "bulk copies move multiples of 16 bytes");
  static_assert(kPgP * R * 2 % 16 == 0, "16-byte factor rows");
};

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   tc::smem_addr(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(tc::smem_addr(bar))
               : "memory");
}

// four 16-bit values (8 bytes) to float
__device__ __forceinline__ void four_f32(uint2 x, float (&f)[4], __half) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&x.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&x.y));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}
__device__ __forceinline__ void four_f32(uint2 x, float (&f)[4], __nv_bfloat16) {
  f[0] = __uint_as_float(x.x << 16); f[1] = __uint_as_float(x.x & 0xffff0000u);
  f[2] = __uint_as_float(x.y << 16); f[3] = __uint_as_float(x.y & 0xffff0000u);
}

// One halving stage of the transpose-reduce: C entries left, partner at lane ^ O. A lane whose bit O
// is set keeps the upper half of its entries and receives the partner's upper half; the other lane
// keeps the lower half. With one entry left the stage is a plain butterfly add.
template <int C, int O>
__device__ __forceinline__ void tr_stage(float* v, int lane) {
  if constexpr (C > 1) {
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int i = 0; i < C / 2; ++i) {
      const float send = up ? v[i] : v[i + C / 2];
      const float keep = up ? v[i + C / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
    }
  } else {
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
  }
}

// Sums of v[0 .. R-1] over the 32 lanes: lane l returns the sum of entry l >> (5 - log2 R).
template <int R>
__device__ __forceinline__ float transpose_reduce(float (&v)[R], int lane) {
  tr_stage<R, 16>(v, lane);
  tr_stage<(R >= 2 ? R / 2 : 1), 8>(v, lane);
  tr_stage<(R >= 4 ? R / 4 : 1), 4>(v, lane);
  tr_stage<(R >= 8 ? R / 8 : 1), 2>(v, lane);
  tr_stage<(R >= 16 ? R / 16 : 1), 1>(v, lane);
  return v[0];
}

template <int R>
constexpr int tr_shift() { return R == 32 ? 0 : R == 16 ? 1 : 2; }

template <typename T, int R>
__global__ void __launch_bounds__(kPgThreads) paged_decode_kernel(const PagedArgs P) {
  using L = PgLay<R>;
  constexpr int kShift = tr_shift<R>();
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* empty = full + L::kSlots;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc);
  volatile int* merge_flag = abort_flag + 1;
  float* qs = reinterpret_cast<float*>(smem + L::kOffQ);
  float* wm = reinterpret_cast<float*>(smem + L::kOffWm);
  float* wl = reinterpret_cast<float*>(smem + L::kOffWl);
  float* wo = reinterpret_cast<float*>(smem + L::kOffWo);
  const DecodeArgs& a = P.m;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;

  int np = P.n_pages[b];
  if (np < 0 || np > P.max_pages) {
    if (threadIdx.x == 0 && split == 0 && h == 0) record_error(P.err, kCodeDevice, kErrSeqLen, np, b);
    np = np < 0 ? 0 : P.max_pages;
  }
  const int p0 = split * P.pages_per_split;
  const int p1 = min(np, p0 + P.pages_per_split);
  const int cnt = p1 > p0 ? p1 - p0 : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kSlots; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  // this head's query, rotated at q_pos on the RoPE path (float64-derived table), pre-scaled
  if (threadIdx.x < kPgDh) {
    const int d = threadIdx.x;
    const int64_t qoff = ((int64_t)b * P.n_heads + h) * kPgDh;
    float v = load_as_f32(P.q, P.q_dtype, qoff + d);
    if (P.rope) {
      int qp = P.q_pos[b];
      if (qp < 0 || qp >= P.max_pos) {
        if (d == 0 && split == 0) record_error(P.err, kCodeDevice, kErrQueryPos, qp, b);
        qp = qp < 0 ? 0 : int(P.max_pos - 1);
      }
      const int k = d & (kPgDh / 2 - 1);
      const float2 cs = P.rope_tab[(int64_t)qp * (kPgDh / 2) + k];
      const float x0 = load_as_f32(P.q, P.q_dtype, qoff + k);
      const float x1 = load_as_f32(P.q, P.q_dtype, qoff + k + kPgDh / 2);
      v = d < kPgDh / 2 ? x0 * cs.x - x1 * cs.y : x1 * cs.x + x0 * cs.y;
    }
    qs[d] = v * P.qscale;
  }
  __syncthreads();

  const int64_t stride = (int64_t)P.n_heads * L::kRec;   // bytes between a head's consecutive pages
  if (warp == 0) {
    // ---------------------------------------------------------------- page-record producer
    if (lane == 0 && cnt > 0) {
      const char* base = static_cast<const char*>(P.pages) + (((int64_t)b * P.capacity + p0) * P.n_heads + h) * L::kRec;
      int issued = 0;
      for (int j = 0; j < cnt; ++j) {
        const int slot = j % L::kSlots;
        const uint32_t round = uint32_t(j / L::kSlots);
        if (!tc::mbar_wait_bounded(&empty[slot], (round & 1) ^ 1, abort_flag, P.wait_ns)) break;
        tc::mbar_arrive_expect_tx(&full[slot], L::kRec);
        bulk_load(smem + slot * L::kRec, base + j * stride, L::kRec, &full[slot]);
        ++issued;
      }
      if (issued < cnt) {
        // drain the copies still in flight before the CTA may exit
        volatile int quiet = 0;
        for (int j = (issued > L::kSlots ? issued - L::kSlots : 0); j < issued; ++j)
          tc::mbar_wait_bounded(&full[j % L::kSlots], uint32_t(j / L::kSlots) & 1, &quiet, P.wait_ns / 10);
      }
    }
  } else {
    // ---------------------------------------------------------------- consumer warps
    const int cw = warp - 1;
    float q4[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) q4[c] = qs[4 * lane + c];
    float m_run = -INFINITY, l_part = 0.f;
    float o4[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = cw; j < cnt; j += kPgWarps) {
      const int slot = j % L::kSlots;
      const bool got = tc::mbar_wait_bounded(&full[slot], uint32_t(j / L::kSlots) & 1, abort_flag, P.wait_ns);
      if (!__all_sync(0xffffffffu, got)) break;   // the flag is set: every role stops
      const uint8_t* rec = smem + slot * L::kRec;
      // u = R_K q
      float v[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float f[4];
        four_f32(*reinterpret_cast<const uint2*>(rec + L::kRK + r * (kPgDh * 2) + lane * 8), f, T{});
        v[r] = fmaf(q4[0], f[0], fmaf(q4[1], f[1], fmaf(q4[2], f[2], q4[3] * f[3])));
      }
      const float u_mine = transpose_reduce<R>(v, lane);
      // s_t = L_K[t] u for this lane's token
      float s = 0.f;
#pragma unroll
      for (int r4 = 0; r4 < R; r4 += 4) {
        float f[4];
        four_f32(*reinterpret_cast<const uint2*>(rec + L::kLK + lane * (R * 2) + r4 * 2), f, T{});
#pragma unroll
        for (int e = 0; e < 4; ++e) s = fmaf(f[e], __shfl_sync(0xffffffffu, u_mine, (r4 + e) << kShift), s);
      }
      // online softmax (base 2)
      const float mn = fmaxf(m_run, warp_max(s));
      const float alpha = exp2f(m_run - mn);   // 0 before the first page (m_run = -inf)
      const float p = exp2f(s - mn);
      l_part = fmaf(l_part, alpha, p);
      m_run = mn;
      // w = p L_V
#pragma unroll
      for (int r4 = 0; r4 < R; r4 += 4) {
        float f[4];
        four_f32(*reinterpret_cast<const uint2*>(rec + L::kLV + lane * (R * 2) + r4 * 2), f, T{});
#pragma unroll
        for (int e = 0; e < 4; ++e) v[r4 + e] = p * f[e];
      }
      const float w_mine = transpose_reduce<R>(v, lane);
      // o = o alpha + w R_V
#pragma unroll
      for (int c = 0; c < 4; ++c) o4[c] *= alpha;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float wr = __shfl_sync(0xffffffffu, w_mine, r << kShift);
        float f[4];
        four_f32(*reinterpret_cast<const uint2*>(rec + L::kRV + r * (kPgDh * 2) + lane * 8), f, T{});
#pragma unroll
        for (int c = 0; c < 4; ++c) o4[c] = fmaf(wr, f[c], o4[c]);
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[slot]);
    }
    const float l_w = warp_sum(l_part);
    if (lane == 0) {
      wm[cw] = m_run;
      wl[cw] = l_w;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) wo[cw * kPgDh + 4 * lane + c] = o4[c];
  }
  __syncthreads();

  // merge the eight warps' states into this split's partial
  if (threadIdx.x < kPgDh) {
    const int d = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kPgWarps; ++w) M = fmaxf(M, wm[w]);
    float Ls = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < kPgWarps; ++w) {
      const float e = wm[w] == -INFINITY ? 0.f : exp2f(wm[w] - M);
      Ls = fmaf(wl[w], e, Ls);
      o = fmaf(wo[w * kPgDh + d], e, o);
    }
    const int64_t bh = (int64_t)b * P.n_heads + h;
    a.part_o[(bh * a.n_splits + split) * kPgDh + d] = o;
    if (d == 0) a.part_ml[bh * a.n_splits + split] = make_float2(M, Ls);
  }
  if (threadIdx.x == 0 && *abort_flag) record_error(P.err, kCodeTimeout, kErrWait, blockIdx.x, b);
  merge_if_last(a, b, h, 1, merge_flag, reinterpret_cast<float*>(smem));   // the ring is free by now
}

template <typename T, int R>
cudaError_t launch_typed(const PagedArgs& P, cudaStream_t st) {
  using L = PgLay<R>;
  auto kern = paged_decode_kernel<T, R>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)P.m.n_splits, (unsigned)P.n_heads, (unsigned)P.m.batch);
  kern<<<grid, kPgThreads, L::kSmem, st>>>(P);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_rank(const PagedArgs& P, cudaStream_t st) {
  switch (P.rank) {
    case 8: return launch_typed<T, 8>(P, st);
    case 16: return launch_typed<T, 16>(P, st);
    case 32: return launch_typed<T, 32>(P, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int paged_ctas_per_sm(int rank) { return rank <= 16 ? 2 : 1; }

cudaError_t launch_decode_paged(const PagedArgs& P, cudaStream_t st) {
  if (P.m.batch == 0) return cudaSuccess;
  return P.dtype == kBF16 ? launch_rank<__nv_bfloat16>(P, st) : launch_rank<__half>(P, st);
}

}  // namespace palu
