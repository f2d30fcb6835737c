// Absorbed-mode (non-RoPE) decode attention: an HBM-streaming kernel.
//
// "Palu: KV-Cache Compression With Low-Rank Projection", key-fusion paragraph: with no
// rotation applied to the keys, q K^T = (q B_k^T) H_k^T, so the scores are taken straight
// against the cached latents and nothing is rebuilt. Per head and token that is one dot
// product of length r for the score and r multiply-adds for p H_v: 4 flop per byte of
// latent, far below the ridge point, so the kernel is bound by HBM and is written as a
// TMA stream feeding CUDA cores.
//
// Per CTA: one (batch row b, group g, T-split) unit, all s = 4 heads of the group.
//   * warp 8 streams 64-token stages of H_k,g and H_v,g (whole 512-byte rows, TMA) through
//     a 3-stage ring (192 KB in flight);
//   * warps 0-7 each take 8 tokens of every stage and keep their own online softmax; a lane
//     owns 8 of the r columns: it holds those columns of the four absorbed queries in
//     registers, forms 32 partial dot products (8 tokens x 4 heads) per stage and finishes
//     them with one transpose-reduction across the warp, then accumulates p H_v for the
//     same columns;
//   * the eight warps' (m, l, o) are merged by log-sum-exp at the end of the CTA.
// Waits are bounded (PALU_ERR_TIMEOUT through the workspace error word).
#include <cuda.h>

#include <mutex>

#include "internal.h"
#include "split_merge.cuh"
#include "tc_ptx.cuh"

namespace palu {

namespace {

constexpr int kHeads = 4;                      // heads per group (s)
constexpr int kRank = 256;                     // r_k = r_v
constexpr int kStageTok = 64;                  // tokens per stage
constexpr int kWarps = 8;                      // compute warps
constexpr int kTokPerWarp = kStageTok / kWarps;  // 8
constexpr int kStages = 3;
constexpr int kRowBytes = kRank * 2;           // 512
constexpr int kHalfStage = kStageTok * kRowBytes;  // 32 KB (K or V)
constexpr int kStageBytes = 2 * kHalfStage;    // 64 KB
constexpr int kThreads = (kWarps + 1) * 32;
constexpr uint64_t kWaitNs = 1000000000ull;   // 1 s per wait

constexpr int kOffRing = 0;
constexpr int kOffBar = kOffRing + kStages * kStageBytes;
constexpr int kOffMisc = kOffBar + 8 * (2 * kStages);
constexpr int kOffP = (kOffMisc + 16 + 15) & ~15;        // float [kWarps][32] per-warp p scratch
constexpr int kOffM = kOffP + kWarps * 32 * 4;          // float [kWarps][kHeads] running max
constexpr int kOffL = kOffM + kWarps * kHeads * 4;      // float [kWarps][kHeads] running sum
constexpr int kSmemBytes = kOffL + kWarps * kHeads * 4;
constexpr int kSmemAlloc = kSmemBytes + 128;
constexpr int kOffO = kOffRing;                          // float [kWarps][kHeads][kRank], reuses the ring
static_assert(kWarps * kHeads * kRank * 4 <= kStages * kStageBytes, "merge buffer fits the ring");
static_assert(kSmemAlloc <= 232448, "shared memory budget");

template <typename T>
__device__ __forceinline__ void unpack8(const uint4& u, float* h);
template <>
__device__ __forceinline__ void unpack8<__half>(const uint4& u, float* h) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    h[2 * i] = f.x;
    h[2 * i + 1] = f.y;
  }
}
template <>
__device__ __forceinline__ void unpack8<__nv_bfloat16>(const uint4& u, float* h) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[2 * i] = __uint_as_float(w[i] << 16);
    h[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Sum 32 per-lane values v[0..31] across the warp so that lane L ends with sum_lanes v[L]
// (transpose-reduction: 31 shuffles and adds for 32 sums).
__device__ __forceinline__ float transpose_reduce32(float* v, int lane) {
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool upper = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      // keep v[i + half] (upper lanes) or v[i] (lower lanes); send the other to the partner
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, half);
    }
  }
  return v[0];
}

template <typename ET>
__global__ void __launch_bounds__(kThreads, 1)
    decode_abs_kernel(const __grid_constant__ CUtensorMap tm_hk, const __grid_constant__ CUtensorMap tm_hv,
                      const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc);
  float* pw = reinterpret_cast<float*>(smem + kOffP);
  float* mw = reinterpret_cast<float*>(smem + kOffM);
  float* lw = reinterpret_cast<float*>(smem + kOffL);
  float* ow = reinterpret_cast<float*>(smem + kOffO);

  int T = a.seq_lens[b];
  if (T < 0 || T > a.max_seq_len) {
    if (threadIdx.x == 0 && split == 0 && g == 0) record_error(a.err, kCodeDevice, kErrSeqLen, T, b);
    T = T < 0 ? 0 : a.max_seq_len;
  }
  const int span = a.tiles_per_split * kStageTok;
  const int t_begin = split * span;
  const int t_end = min(T, t_begin + span);
  const int n_stages = t_end > t_begin ? (t_end - t_begin + kStageTok - 1) / kStageTok : 0;
  const int head0 = g * kHeads;
  const int cache_g = a.g_split > 1 ? g / a.g_split : g;   // split groups share their cache group's latents

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], kWarps);
    }
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_stages > 0) {
      tc::tma_prefetch(&tm_hk);
      tc::tma_prefetch(&tm_hv);
      const int row0 = b * (int)a.capacity;
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < n_stages && ok; ++i) {
        const int s = i % kStages;
        if (!tc::mbar_wait_bounded(&empty[s], ((i / kStages) & 1) ^ 1, abort_flag, kWaitNs)) {
          ok = false;
          break;
        }
        tc::mbar_arrive_expect_tx(&full[s], kStageBytes);
        const int r = row0 + t_begin + i * kStageTok;
        tc::tma_load_3d(smem + kOffRing + s * kStageBytes, &tm_hk, &full[s], 0, cache_g, r);
        tc::tma_load_3d(smem + kOffRing + s * kStageBytes + kHalfStage, &tm_hv, &full[s], 0, cache_g, r);
        ++issued;
      }
      if (!ok) {
        volatile int quiet = 0;
        for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
          tc::mbar_wait_bounded(&full[i % kStages], (i / kStages) & 1, &quiet, kWaitNs / 10);
      }
    }
  } else {
    // ------------------------------------------------------------ compute warps
    // absorbed queries of the four heads for this lane's columns (pre-scaled by log2(e)/sqrt(d_h))
    float q[kHeads][8];
#pragma unroll
    for (int j = 0; j < kHeads; ++j) {
      const float4* src = reinterpret_cast<const float4*>(a.qbuf + ((int64_t)b * a.n_heads + head0 + j) * kRank +
                                                          lane * 8);
      const float4 x = src[0], y = src[1];
      q[j][0] = x.x; q[j][1] = x.y; q[j][2] = x.z; q[j][3] = x.w;
      q[j][4] = y.x; q[j][5] = y.y; q[j][6] = y.z; q[j][7] = y.w;
    }
    float acc[kHeads][8];
#pragma unroll
    for (int j = 0; j < kHeads; ++j)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[j][c] = 0.f;
    float m_run[kHeads] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    float l_run = 0.f;   // running sum of head (lane & 3) over this warp's tokens
    // ALiBi: this lane's head (lane & 3) adds m (pos_t - q_pos) log2(e) to its scores
    float alibi_m = 0.f, alibi_qp = 0.f;
    if (a.alibi) {
      alibi_m = exp2f(-8.f * float(head0 + (lane & 3) + 1) / float(a.n_heads)) * 1.4426950408889634f;
      int qp = T > 0 ? (a.positions ? a.positions[(int64_t)b * a.capacity + T - 1] : T - 1) : 0;
      if (a.q_pos) qp = a.q_pos[b];
      alibi_qp = float(qp);
    }
    bool broken = false;
    float* myp = pw + warp * 32;

    for (int i = 0; i < n_stages; ++i) {
      const int s = i % kStages;
      if (!tc::mbar_wait_bounded(&full[s], (i / kStages) & 1, abort_flag, kWaitNs)) broken = true;
      if (broken) {
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[s]);
        continue;
      }
      const uint8_t* kst = smem + kOffRing + s * kStageBytes + (warp * kTokPerWarp) * kRowBytes + lane * 16;
      const uint8_t* vst = kst + kHalfStage;
      const int tok0 = t_begin + i * kStageTok + warp * kTokPerWarp;

      // partial scores: 8 tokens x 4 heads over this lane's 8 columns
      float part[32];
#pragma unroll
      for (int t = 0; t < kTokPerWarp; ++t) {
        float h[8];
        unpack8<ET>(*reinterpret_cast<const uint4*>(kst + t * kRowBytes), h);
#pragma unroll
        for (int j = 0; j < kHeads; ++j) {
          float sacc = q[j][0] * h[0];
#pragma unroll
          for (int c = 1; c < 8; ++c) sacc = fmaf(q[j][c], h[c], sacc);
          part[t * kHeads + j] = sacc;
        }
      }
      // lane L now owns the score of token L / 4, head L % 4
      float sc = transpose_reduce32(part, lane);
      const int jl = lane & 3;
      const int tk = tok0 + (lane >> 2);
      if (a.alibi && tk < t_end) {
        const int pos = a.positions ? a.positions[(int64_t)b * a.capacity + tk] : tk;
        sc = fmaf(alibi_m, float(pos) - alibi_qp, sc);
      }
      if (tk >= t_end) sc = -INFINITY;

      // online softmax per head over this warp's tokens
      float bm = sc;
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
      float alpha[kHeads], mnew[kHeads];
#pragma unroll
      for (int j = 0; j < kHeads; ++j) {
        const float bmj = __shfl_sync(0xffffffffu, bm, j);
        mnew[j] = fmaxf(m_run[j], bmj);
        alpha[j] = (mnew[j] == -INFINITY) ? 1.f : exp2f(m_run[j] - mnew[j]);
        m_run[j] = mnew[j];
      }
      // this lane's head jl (register selects, no dynamically indexed arrays)
      const float m_l = jl == 0 ? mnew[0] : jl == 1 ? mnew[1] : jl == 2 ? mnew[2] : mnew[3];
      const float a_l = jl == 0 ? alpha[0] : jl == 1 ? alpha[1] : jl == 2 ? alpha[2] : alpha[3];
      const float p = (sc == -INFINITY) ? 0.f : exp2f(sc - m_l);
      float ps = p;
      ps += __shfl_xor_sync(0xffffffffu, ps, 4);
      ps += __shfl_xor_sync(0xffffffffu, ps, 8);
      ps += __shfl_xor_sync(0xffffffffu, ps, 16);
      l_run = l_run * a_l + ps;
      myp[lane] = p;
      __syncwarp();

      // p H_v for this lane's 8 columns
#pragma unroll
      for (int j = 0; j < kHeads; ++j)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[j][c] *= alpha[j];
#pragma unroll
      for (int t = 0; t < kTokPerWarp; ++t) {
        if (tok0 + t >= t_end) break;   // rows past the sequence may hold anything
        float h[8];
        unpack8<ET>(*reinterpret_cast<const uint4*>(vst + t * kRowBytes), h);
        const float4 p4 = *reinterpret_cast<const float4*>(myp + t * kHeads);
        const float pv[kHeads] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
        for (int j = 0; j < kHeads; ++j)
#pragma unroll
          for (int c = 0; c < 8; ++c) acc[j][c] = fmaf(pv[j], h[c], acc[j][c]);
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[s]);
    }

    // merge the eight warps: (m, l) per head, o per head and column
    const bool aborted = tc::named_bar_or(1, kWarps * 32, broken || *abort_flag != 0);
    if (!aborted) {
      if (lane < kHeads) {
        mw[warp * kHeads + lane] = m_run[lane];
        lw[warp * kHeads + lane] = l_run;   // lane j holds head j's sum
      }
#pragma unroll
      for (int j = 0; j < kHeads; ++j)
#pragma unroll
        for (int c = 0; c < 8; ++c) ow[(warp * kHeads + j) * kRank + lane * 8 + c] = acc[j][c];
      tc::named_bar(1, kWarps * 32);
      const int tid = threadIdx.x;
      for (int idx = tid; idx < kHeads * kRank; idx += kWarps * 32) {
        const int j = idx / kRank, c = idx % kRank;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mw[w * kHeads + j]);
        float o = 0.f, L = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float mwj = mw[w * kHeads + j];
          const float f = (mwj == -INFINITY) ? 0.f : exp2f(mwj - M);
          o = fmaf(ow[(w * kHeads + j) * kRank + c], f, o);
          L = fmaf(lw[w * kHeads + j], f, L);
        }
        const int64_t bh = (int64_t)b * a.n_heads + head0 + j;
        a.part_o[(bh * a.n_splits + split) * kRank + c] = o;
        if (c == 0) a.part_ml[bh * a.n_splits + split] = make_float2(M, L);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) record_error(a.err, kCodeTimeout, kErrWait, blockIdx.x, b);
  merge_if_last(a, b, head0, kHeads, reinterpret_cast<volatile int*>(smem + kOffMisc + 4),
                reinterpret_cast<float*>(smem + kOffRing));  // the ring is free by now
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

bool abs_supported(const DecodeArgs& a) {
  return (a.k_dtype == kF16 || a.k_dtype == kBF16) && a.v_dtype == a.k_dtype && a.s == kHeads && a.rk == kRank &&
         a.rv == kRank && (int64_t)a.batch * a.capacity >= kStageTok &&
         (int64_t)a.batch * a.capacity < (int64_t(1) << 31) && encode_fn() != nullptr;
}

int abs_stage_tokens() { return kStageTok; }

cudaError_t launch_decode_abs(const DecodeArgs& a, cudaStream_t st) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const CUtensorMapDataType dt = a.k_dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap tm[2];
  const void* base[2] = {a.hk, a.hv};
  for (int i = 0; i < 2; ++i) {
    // the cache's own groups: split groups (g_split > 1) share one cache group
    const int cache_n_g = a.g_split > 1 ? a.n_g / a.g_split : a.n_g;
    const cuuint64_t dims[3] = {(cuuint64_t)kRank, (cuuint64_t)cache_n_g, (cuuint64_t)a.batch * a.capacity};
    const cuuint64_t strides[2] = {(cuuint64_t)kRank * 2, (cuuint64_t)cache_n_g * kRank * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kRank, 1, (cuuint32_t)kStageTok};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tm[i], dt, 3, const_cast<void*>(base[i]), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  dim3 grid(a.n_splits, a.n_g, a.batch);
  cudaError_t e;
  if (a.k_dtype == kBF16) {
    e = cudaFuncSetAttribute(decode_abs_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    decode_abs_kernel<__nv_bfloat16><<<grid, kThreads, kSmemAlloc, st>>>(tm[0], tm[1], a);
  } else {
    e = cudaFuncSetAttribute(decode_abs_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    decode_abs_kernel<__half><<<grid, kThreads, kSmemAlloc, st>>>(tm[0], tm[1], a);
  }
  return cudaGetLastError();
}

}  // namespace palu
