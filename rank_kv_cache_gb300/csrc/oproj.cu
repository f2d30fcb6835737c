// The layer's output projection over the latent decode outputs, with B_v fused into W_o.
//
// "Palu: KV-Cache Compression With Low-Rank Projection", method section, value-fusion
// paragraph: head i's attention output is p_i V_i = p_i H_v,g B_v^(i), and it only ever meets
// its own rows W_o^(i) of the output projection, so the value latents are never rebuilt:
//   y[b] = sum_i o[b][i] W_f^(i),   W_f^(i) = B_v^(i) W_o^(i)   (r_v x d per head),
// with o = p H_v the decode kernels' output. The fused weight stacks the heads' blocks as
// [n r_v][d]: twice the size of W_o when r_v = 2 d_h (the Llama-2-7B shapes, 64 MB in fp16).
//
// * fuse_vo_kernel forms W_f once (an offline transform): fp32 accumulation, rounded once.
// * oproj_kernel is the per-step GEMV y = o W_f. Every weight element is read once and used
//   NB times (NB = batch rows per launch block, <= 8), so the kernel is bound by HBM and is
//   written as a stream of 16-byte non-allocating loads, 8 or 16 rows in flight per thread,
//   feeding packed f32x2 FMAs. A CTA owns 128 columns of one K chunk: 16 column lanes x 16
//   row groups interleaved over the chunk's rows. Row groups are reduced by a shuffle and
//   through shared memory; the chunk partials of a column block are summed in a fixed order by
//   the last CTA to finish that block (an atomic counter it resets), so results are
//   deterministic and a call is one launch.
#include <mutex>

#include "palu_attn.h"
#include "internal.h"

namespace palu {
namespace {

constexpr int kOpThreads = 256;
constexpr int kOpColLanes = 16;                     // threads across a CTA's columns
constexpr int kOpCols = kOpColLanes * 8;            // 128 columns per CTA
constexpr int kOpKSub = kOpThreads / kOpColLanes;   // 16 interleaved row groups
// rows in flight per thread: 16 for four batch rows, 8 otherwise (measured on GB300: with 16, the
// four-row GEMV ran 22 us instead of 29 us, the one- and eight-row ones slower)
template <int NB>
constexpr int op_unroll() { return NB == 4 ? 16 : 8; }
template <int NB>
constexpr int op_row_quantum() { return kOpKSub * op_unroll<NB>(); }   // chunk rows are a multiple of this
constexpr int kOpMaxChunkRows = 1024;
constexpr int kOpMaxChunks = 64;
constexpr int kOpMaxNB = 8;
constexpr int kOpMaxBatch = 1024;                   // n_bb <= kOpMaxBatch / kOpMaxNB
constexpr int64_t kOpMaxK = (int64_t)kOpMaxChunks * kOpMaxChunkRows;

struct OprojArgs {
  const void* w;         // [K][d] fp16 / bf16
  const float* o;        // [batch][K]
  float* y;              // [batch][d]
  float* part;           // [n_chunks][batch][d]
  unsigned* counters;    // [n_bb][n_cb], zero between calls
  int64_t K, d;
  int batch, kc, n_chunks, n_cb;
};

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void w8_to_float2x4(const uint4& u, float2* f, __half) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) f[j] = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
}
__device__ __forceinline__ void w8_to_float2x4(const uint4& u, float2* f, __nv_bfloat16) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) f[j] = make_float2(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xffff0000u));
}

template <typename WT, int NB>
__global__ void __launch_bounds__(kOpThreads) oproj_kernel(const OprojArgs p) {
  extern __shared__ __align__(16) float sm[];
  float* os = sm;                                   // [kc][NB]: the chunk's o values
  float* red = sm + p.kc * NB;                      // [8 warps][NB][kOpCols]
  __shared__ int last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cb = blockIdx.x, chunk = blockIdx.y, bb = blockIdx.z;
  const int b0 = bb * NB;
  const int64_t k0 = (int64_t)chunk * p.kc;
  const int rows = (int)min((int64_t)p.kc, p.K - k0);
  const int c8 = tid % kOpColLanes, ks = tid / kOpColLanes;
  const int64_t col = (int64_t)cb * kOpCols + c8 * 8;
  const bool cvalid = col < p.d;   // d is a multiple of 8: a lane's 8 columns are all in or all out
  const WT* wp = static_cast<const WT*>(p.w) + k0 * p.d + col;
  float2 acc[NB][4];
#pragma unroll
  for (int bi = 0; bi < NB; ++bi)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[bi][c] = make_float2(0.f, 0.f);

  // rows ks, ks + 16, ...: every row index below stays inside the chunk's kc rows (kc is a
  // multiple of the row quantum), and rows past the end of K load nothing and meet o = 0
  constexpr int kOpUnroll = op_unroll<NB>(), kOpRowQuantum = op_row_quantum<NB>();
  uint4 u[kOpUnroll];
  auto load_rows = [&](int r0) {
#pragma unroll
    for (int q = 0; q < kOpUnroll; ++q) {
      const int r = r0 + q * kOpKSub;
      u[q] = (cvalid && r < rows) ? ld_stream16(wp + (int64_t)r * p.d) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  // For one or two batch rows the first rows of weights are requested before o is staged (they
  // do not depend on it), which hides the staging's latency (b1: 26 -> 20 us on GB300). With more
  // batch rows the registers held across the staging cost more than they save.
  constexpr bool kEarly = NB <= 2;
  if (kEarly) load_rows(ks);
  for (int i = tid; i < p.kc * NB; i += kOpThreads) {
    const int k = i / NB, bi = i % NB;
    os[i] = (k < rows && b0 + bi < p.batch) ? p.o[(int64_t)(b0 + bi) * p.K + k0 + k] : 0.f;
  }
  __syncthreads();

  for (int r0 = ks; r0 < rows; r0 += kOpRowQuantum) {
    if (!kEarly || r0 != ks) load_rows(r0);
#pragma unroll
    for (int q = 0; q < kOpUnroll; ++q) {
      const int r = r0 + q * kOpKSub;
      float2 f[4];
      w8_to_float2x4(u[q], f, WT{});
      float ov[NB];
      if constexpr (NB % 4 == 0) {
#pragma unroll
        for (int v = 0; v < NB / 4; ++v) {
          const float4 x = reinterpret_cast<const float4*>(os + r * NB)[v];
          ov[4 * v] = x.x; ov[4 * v + 1] = x.y; ov[4 * v + 2] = x.z; ov[4 * v + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int bi = 0; bi < NB; ++bi) ov[bi] = os[r * NB + bi];
      }
#pragma unroll
      for (int bi = 0; bi < NB; ++bi) {
        const float2 o2 = make_float2(ov[bi], ov[bi]);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[bi][c] = __ffma2_rn(o2, f[c], acc[bi][c]);
      }
    }
  }

  // row groups 2w and 2w + 1 share warp w (lanes 0-15 / 16-31): add them with one shuffle, then
  // reduce the eight warps through shared memory
#pragma unroll
  for (int bi = 0; bi < NB; ++bi)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      acc[bi][c].x += __shfl_xor_sync(0xffffffffu, acc[bi][c].x, 16);
      acc[bi][c].y += __shfl_xor_sync(0xffffffffu, acc[bi][c].y, 16);
    }
  if (lane < kOpColLanes) {
#pragma unroll
    for (int bi = 0; bi < NB; ++bi) {
      float4* dst = reinterpret_cast<float4*>(red + (warp * NB + bi) * kOpCols + c8 * 8);
      dst[0] = make_float4(acc[bi][0].x, acc[bi][0].y, acc[bi][1].x, acc[bi][1].y);
      dst[1] = make_float4(acc[bi][2].x, acc[bi][2].y, acc[bi][3].x, acc[bi][3].y);
    }
  }
  __syncthreads();
  const bool single = p.n_chunks == 1;
  for (int idx = tid; idx < NB * kOpCols; idx += kOpThreads) {
    const int bi = idx / kOpCols, c = idx % kOpCols;
    const int64_t cc = (int64_t)cb * kOpCols + c;
    const int b = b0 + bi;
    if (cc >= p.d || b >= p.batch) continue;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kOpThreads / 32; ++w) s += red[(w * NB + bi) * kOpCols + c];
    if (single) p.y[(int64_t)b * p.d + cc] = s;
    else p.part[((int64_t)chunk * p.batch + b) * p.d + cc] = s;
  }
  if (single) return;

  // the last CTA of this (batch block, column block) sums the chunk partials in chunk order
  __threadfence();
  __syncthreads();
  unsigned* ctr = p.counters + (int64_t)bb * p.n_cb + cb;
  if (tid == 0) last = (atomicAdd(ctr, 1u) == unsigned(p.n_chunks - 1)) ? 1 : 0;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // The chunk partials of the block are requested eight at a time per thread,
  // then summed in chunk order: the order, and so the result, does not depend on the timing.
  for (int idx = tid; idx < NB * kOpCols; idx += kOpThreads) {
    const int bi = idx / kOpCols, c = idx % kOpCols;
    const int64_t cc = (int64_t)cb * kOpCols + c;
    const int b = b0 + bi;
    if (cc >= p.d || b >= p.batch) continue;
    const float* pp = p.part + (int64_t)b * p.d + cc;
    const int64_t stride = (int64_t)p.batch * p.d;
    float s = 0.f;
    for (int ch0 = 0; ch0 < p.n_chunks; ch0 += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = ch0 + j < p.n_chunks ? __ldcg(pp + (ch0 + j) * stride) : 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) s += v[j];
    }
    p.y[(int64_t)b * p.d + cc] = s;
  }
  if (tid == 0) *ctr = 0u;
}

// W_f[i r_v + m][c] = sum_e B_v[g][m][j d_h + e] W_o[i d_h + e][c] (g = i / s, j = i % s), fp32
// accumulation over e in the order e = 0 .. d_h - 1, rounded once to the output dtype.
// Tiles of 64 x 64 outputs per 256-thread block (4 x 4 per thread), 16-deep slices of e staged
// in shared memory.
template <typename IT, typename OT>
__global__ void __launch_bounds__(256) fuse_vo_kernel(const IT* __restrict__ bv, const IT* __restrict__ wo,
                                                      OT* __restrict__ wf, int s, int dh, int rv, int64_t d) {
  __shared__ float As[16][64 + 1];   // [e][m]
  __shared__ float Bs[16][64];       // [e][c]
  const int i = blockIdx.z, g = i / s, j = i % s;
  const int m0 = blockIdx.y * 64;
  const int64_t c0 = (int64_t)blockIdx.x * 64;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int e0 = 0; e0 < dh; e0 += 16) {
    for (int t = threadIdx.x; t < 16 * 64; t += 256) {
      const int e = t % 16, m = t / 16;
      As[e][m] = (m0 + m < rv && e0 + e < dh)
                     ? to_f32(bv[((int64_t)g * rv + m0 + m) * (int64_t)(s * dh) + j * dh + e0 + e])
                     : 0.f;
      const int c = t % 64, e2 = t / 64;
      Bs[e2][c] = (c0 + c < d && e0 + e2 < dh) ? to_f32(wo[((int64_t)i * dh + e0 + e2) * d + c0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        a[u] = As[e][ty * 4 + u];
        b[u] = Bs[e][tx * 4 + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], b[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int m = m0 + ty * 4 + u;
    if (m >= rv) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int64_t c = c0 + tx * 4 + v;
      if (c < d) wf[((int64_t)i * rv + m) * d + c] = from_f32<OT>(acc[u][v]);
    }
  }
}

template <typename IT>
cudaError_t launch_fuse_typed(const void* bv, const void* wo, int out_dtype, void* wf, int n, int s, int dh, int rv,
                              int64_t d, cudaStream_t st) {
  dim3 grid((unsigned)((d + 63) / 64), (unsigned)((rv + 63) / 64), (unsigned)n);
  const IT* b = static_cast<const IT*>(bv);
  const IT* w = static_cast<const IT*>(wo);
  if (out_dtype == kBF16)
    fuse_vo_kernel<IT, __nv_bfloat16><<<grid, 256, 0, st>>>(b, w, static_cast<__nv_bfloat16*>(wf), s, dh, rv, d);
  else
    fuse_vo_kernel<IT, __half><<<grid, 256, 0, st>>>(b, w, static_cast<__half*>(wf), s, dh, rv, d);
  return cudaGetLastError();
}

size_t oproj_smem(int kc, int nb) { return (size_t)kc * nb * 4 + (size_t)(kOpThreads / 32) * nb * kOpCols * 4; }

template <typename WT, int NB>
cudaError_t launch_oproj_nb(const OprojArgs& a0, int n_bb, int sm_count, cudaStream_t st) {
  OprojArgs a = a0;
  auto kern = oproj_kernel<WT, NB>;
  const size_t smem_max = oproj_smem(kOpMaxChunkRows, NB);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kOpThreads, smem_max);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  // as many K chunks as fill one wave of CTAs, within [ceil(K / 1024), min(64, ceil(K / 128))]
  const int64_t slots = (int64_t)sm_count * per_sm;
  int64_t want = slots / ((int64_t)a.n_cb * n_bb);
  const int64_t lo = (a.K + kOpMaxChunkRows - 1) / kOpMaxChunkRows;
  constexpr int kOpRowQuantum = op_row_quantum<NB>();
  int64_t hi = (a.K + kOpRowQuantum - 1) / kOpRowQuantum;
  if (hi > kOpMaxChunks) hi = kOpMaxChunks;
  if (want > hi) want = hi;
  if (want < lo) want = lo;
  if (want < 1) want = 1;
  int64_t kc = (a.K + want - 1) / want;
  kc = (kc + kOpRowQuantum - 1) / kOpRowQuantum * kOpRowQuantum;
  a.kc = (int)kc;
  a.n_chunks = (int)((a.K + kc - 1) / kc);
  dim3 grid((unsigned)a.n_cb, (unsigned)a.n_chunks, (unsigned)n_bb);
  kern<<<grid, kOpThreads, oproj_smem(a.kc, NB), st>>>(a);
  return cudaGetLastError();
}

template <typename WT>
cudaError_t launch_oproj_typed(const OprojArgs& a, int sm_count, cudaStream_t st) {
  const int nb = a.batch >= 8 ? 8 : a.batch >= 4 ? 4 : a.batch >= 2 ? 2 : 1;
  const int n_bb = (a.batch + nb - 1) / nb;
  switch (nb) {
    case 8: return launch_oproj_nb<WT, 8>(a, n_bb, sm_count, st);
    case 4: return launch_oproj_nb<WT, 4>(a, n_bb, sm_count, st);
    case 2: return launch_oproj_nb<WT, 2>(a, n_bb, sm_count, st);
    default: return launch_oproj_nb<WT, 1>(a, n_bb, sm_count, st);
  }
}

// workspace: counters [kOpMaxBatch / kOpMaxNB][n_cb] at a fixed offset (so that calls with
// different batch sizes find the same, zeroed counters), then partials [kOpMaxChunks][batch][d]
size_t oproj_counter_bytes(int64_t d) {
  const int64_t n_cb = (d + kOpCols - 1) / kOpCols;
  return ((size_t)(kOpMaxBatch / kOpMaxNB) * n_cb * sizeof(unsigned) + 255) & ~size_t(255);
}
size_t oproj_ws_bytes(int64_t d, int max_batch) {
  return oproj_counter_bytes(d) + (size_t)kOpMaxChunks * max_batch * d * sizeof(float);
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices];

// the calling thread's current device and its SM count; the stream must belong to it
palu_status_t current_device(palu_stream_t stream, int* sms) {
  int dev = 0, sdev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PALU_ERR_CUDA;
  if (cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) {
    cudaGetLastError();
    return PALU_ERR_INVALID_ARG;
  }
  if (sdev != dev) return PALU_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[dev] && cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PALU_ERR_CUDA;
  *sms = g_sms[dev];
  return PALU_OK;
}

}  // namespace
}  // namespace palu

using namespace palu;

extern "C" {

palu_status_t palu_fuse_value_output(const void* B_v, const void* W_o, palu_dtype_t in_dtype, int n_heads,
                                     int head_dim, int group_size, int rank_v, int64_t d_model, void* W_fused,
                                     palu_dtype_t out_dtype, palu_stream_t stream) {
  if (!B_v || !W_o || !W_fused) return PALU_ERR_INVALID_ARG;
  if ((unsigned)in_dtype > PALU_BF16 || (out_dtype != PALU_F16 && out_dtype != PALU_BF16)) return PALU_ERR_INVALID_ARG;
  if (n_heads <= 0 || head_dim <= 0 || group_size <= 0 || n_heads % group_size || rank_v <= 0 || d_model <= 0)
    return PALU_ERR_INVALID_ARG;
  const size_t ie = in_dtype == PALU_F32 ? 4 : 2;
  if ((uintptr_t)B_v % ie || (uintptr_t)W_o % ie || (uintptr_t)W_fused % 2) return PALU_ERR_INVALID_ARG;
  int sms = 0;
  const palu_status_t st = current_device(stream, &sms);
  if (st != PALU_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (in_dtype == PALU_F32)
    e = launch_fuse_typed<float>(B_v, W_o, out_dtype, W_fused, n_heads, group_size, head_dim, rank_v, d_model, s);
  else if (in_dtype == PALU_BF16)
    e = launch_fuse_typed<__nv_bfloat16>(B_v, W_o, out_dtype, W_fused, n_heads, group_size, head_dim, rank_v,
                                         d_model, s);
  else
    e = launch_fuse_typed<__half>(B_v, W_o, out_dtype, W_fused, n_heads, group_size, head_dim, rank_v, d_model, s);
  return e == cudaSuccess ? PALU_OK : PALU_ERR_CUDA;
}

palu_status_t palu_output_proj_workspace_size(int64_t k_dim, int64_t d_model, int max_batch, size_t* bytes) {
  if (!bytes || k_dim <= 0 || d_model <= 0 || d_model % 8 || max_batch <= 0) return PALU_ERR_INVALID_ARG;
  if (k_dim > kOpMaxK || max_batch > kOpMaxBatch || d_model > (int64_t(1) << 31)) return PALU_ERR_UNSUPPORTED;
  *bytes = oproj_ws_bytes(d_model, max_batch);
  return PALU_OK;
}

palu_status_t palu_output_proj(const void* W_fused, palu_dtype_t w_dtype, int64_t k_dim, int64_t d_model,
                               const float* o, int batch, float* y, void* workspace, size_t workspace_bytes,
                               palu_stream_t stream) {
  if (w_dtype != PALU_F16 && w_dtype != PALU_BF16) return PALU_ERR_INVALID_ARG;
  if (k_dim <= 0 || d_model <= 0 || d_model % 8 || batch < 0) return PALU_ERR_INVALID_ARG;
  if (k_dim > kOpMaxK || batch > kOpMaxBatch || d_model > (int64_t(1) << 31)) return PALU_ERR_UNSUPPORTED;
  if (batch == 0) return PALU_OK;
  if (!W_fused || (uintptr_t)W_fused % 16 || !o || (uintptr_t)o % 4 || !y || (uintptr_t)y % 4)
    return PALU_ERR_INVALID_ARG;
  if (!workspace || (uintptr_t)workspace % 256 || workspace_bytes < oproj_ws_bytes(d_model, batch))
    return PALU_ERR_WORKSPACE;
  int sms = 0;
  const palu_status_t st = current_device(stream, &sms);
  if (st != PALU_OK) return st;
  OprojArgs a{};
  a.w = W_fused;
  a.o = o;
  a.y = y;
  a.counters = static_cast<unsigned*>(workspace);
  a.part = reinterpret_cast<float*>(static_cast<char*>(workspace) + oproj_counter_bytes(d_model));
  a.K = k_dim;
  a.d = d_model;
  a.batch = batch;
  a.n_cb = (int)((d_model + kOpCols - 1) / kOpCols);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = w_dtype == PALU_BF16 ? launch_oproj_typed<__nv_bfloat16>(a, sms, s)
                                             : launch_oproj_typed<__half>(a, sms, s);
  return e == cudaSuccess ? PALU_OK : PALU_ERR_CUDA;
}

}  // extern "C"
