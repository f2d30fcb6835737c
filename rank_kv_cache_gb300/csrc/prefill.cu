// Latent production on tcgen05 tensor cores: H = x A_g for every group of the key and value
// down-projections, written straight into the latent cache.
//
// "Palu: KV-Cache Compression With Low-Rank Projection", method section (SVD rewrite: the layer
// caches h = x A in place of k = x W; G-LRD paragraph: one A_g per group of s heads) and the
// supplementary section (per-token quantisation of the cached latents).
//
// Persistent: one CTA per SM walks the tiles (128 tokens x one side x group), the (side, group)
// index running fastest. Tile t computes D[128 x r] = x_tile[128 x d] W_(side, g)^T, where
// W = [2][n_g][r][d] is A transposed once into the K-major operand (palu_prepare_down_proj).
//   * warp 0 streams 64-column chunks of x (128 rows, 16 KB) and of W (r rows) by TMA with the
//     128-byte swizzle through a 4-stage ring that runs on across the CTA's tiles;
//   * warp 1 issues tcgen05.mma (kind::f16, M = 128, N = r, K = 16; fp32 accumulation in TMEM)
//     into one of two 256-column accumulators, so the MMA of the next tile overlaps the epilogue;
//   * warpgroup 1 (thread = token row, its TMEM lane) reads the finished row back and writes it:
//     fp32, fp16 or bf16 values (round to nearest), or for int4 caches one fp16 scale and r / 2
//     bytes of codes, with the quantiser of the append path (scale = fp16(min(amax / 7, 65504)),
//     code = clamp(rint(h / scale), -7, 7), IEEE division, element 2j in the low nibble), then
//     hands the accumulator back to the MMA warp.
// An int4 row needs the amax over its whole rank, so a tile spans one group's r columns. The
// CTAs work on neighbouring tiles at any time, so a token tile is read from HBM about once and
// the 2 n_g r x d operand stays in L2.
// Every mbarrier wait is bounded; a wait that gives up records PALU_ERR_TIMEOUT in the error word,
// drains the copies it issued and frees TMEM.
#include "internal.h"
#include "tc_ptx.cuh"

namespace palu {
namespace {

constexpr int kPTile = 128;                            // tokens per tile (MMA M)
constexpr int kPChunk = 64;                            // d columns per 128-byte swizzled row
constexpr int kPStages = 4;
constexpr int kPThreads = 256;
constexpr int kPAStage = kPTile * kPChunk * 2;         // 16 KB of x
constexpr int kPBMax = 256 * kPChunk * 2;              // 32 KB of W (r <= 256)
constexpr int kPStageBytes = kPAStage + kPBMax;
constexpr int kPOffBar = kPStages * kPStageBytes;
constexpr int kPSmem = kPOffBar + 128 + 1024;          // barriers, TMEM slot, abort flag; alignment
constexpr uint32_t kPAccCols = 256;                    // one accumulator (N <= 256)
constexpr uint32_t kPTmemCols = 2 * kPAccCols;         // double-buffered

struct PrefillParams {
  ProjectArgs a;
  int bf16;
};

// The int4 code of h for scale sf != 0: clamp(rint(h / sf), -7, 7) with the IEEE quotient, as the
// append path and the oracle take it. h * (1 / sf) is within two units in the last place of
// h / sf (|h / sf| < 8, so within 2^-20), so it rounds to the same integer unless the quotient lies
// within 2^-17 of a half-integer; only then is the correctly rounded division taken.
__device__ __forceinline__ int int4_code_of(float h, float sf, float inv) {
  const float q = h * inv;
  float r = rintf(q);
  if (fabsf(fabsf(q - r) - 0.5f) < 7.62939453125e-06f) r = rintf(__fdiv_rn(h, sf));
  return int(fminf(fmaxf(r, -7.f), 7.f));
}

// one token row of 32 columns from TMEM (columns c0 .. c0 + 31 of this thread's lane)
__device__ __forceinline__ void load_row32(uint32_t taddr, uint32_t (&v)[32]) {
  tc::tmem_ld16x2_nowait(taddr, taddr + 16, v);
  tc::tmem_ld_wait();
}

// Write one finished token row (this thread's TMEM lane, accumulator columns at taddr) into the cache:
// fp32 / fp16 / bf16 values, or int4 codes and their fp16 scale. The TMEM loads are warp-collective, so
// every thread of the warp runs this; only rows with `store` write.
__device__ __forceinline__ void write_row(const ProjectArgs& a, uint32_t taddr, int side, int64_t crow, bool store) {
  uint32_t v[32];
  if (a.cache_dtype == kINT4) {
    float amax = 0.f;
    for (int c0 = 0; c0 < a.rank; c0 += 32) {
      load_row32(taddr + c0, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(__uint_as_float(v[i])));
    }
    const __half sc = __float2half_rn(fminf(__fdiv_rn(amax, 7.0f), 65504.0f));
    const float sf = __half2float(sc);
    const float inv = sf != 0.f ? 1.0f / sf : 0.f;
    uint8_t* out = static_cast<uint8_t*>(a.cache[side]) + crow * (a.rank / 2);
    for (int c0 = 0; c0 < a.rank; c0 += 32) {
      load_row32(taddr + c0, v);
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = sf != 0.f ? int4_code_of(__uint_as_float(v[8 * j + e]), sf, inv) : 0;
          word |= uint32_t(c & 0xF) << (4 * e);
        }
        w[j] = word;
      }
      if (store) *reinterpret_cast<uint4*>(out + c0 / 2) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (store) a.scale[side][crow] = sc;
    return;
  }
  for (int c0 = 0; c0 < a.rank; c0 += 32) {
    load_row32(taddr + c0, v);
    if (!store) continue;
    if (a.cache_dtype == kF32) {
      float4* out = reinterpret_cast<float4*>(static_cast<float*>(a.cache[side]) + crow * a.rank + c0);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        out[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]), __uint_as_float(v[4 * j + 2]),
                             __uint_as_float(v[4 * j + 3]));
    } else {
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float lo = __uint_as_float(v[2 * j]), hi = __uint_as_float(v[2 * j + 1]);
        if (a.cache_dtype == kF16) {
          const __half2 h2 = __floats2half2_rn(lo, hi);
          w[j] = *reinterpret_cast<const uint32_t*>(&h2);
        } else {
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
          w[j] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      }
      uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.cache[side]) + crow * a.rank + c0);
#pragma unroll
      for (int j = 0; j < 4; ++j) out[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    }
  }
}

// Persistent: CTA c takes tiles c, c + gridDim.x, ... (tile = token tile x (side, group), the (side,
// group) index running fastest). The TMA ring runs on across tiles; the MMA of a tile goes into one of
// two TMEM accumulators while the epilogue drains the other.
__global__ void __launch_bounds__(kPThreads, 1)
    project_latents_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                           const PrefillParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const ProjectArgs& a = P.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_nt = 2 * a.n_g;
  const int n_tiles = int((a.M + kPTile - 1) / kPTile) * n_nt;
  const int my_tiles = n_tiles > (int)blockIdx.x ? (n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int nk = int(a.d / kPChunk);
  const uint32_t b_bytes = uint32_t(a.rank) * kPChunk * 2;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPOffBar);
  uint64_t* empty = full + kPStages;
  uint64_t* acc_full = empty + kPStages;     // [2]
  uint64_t* acc_empty = acc_full + 2;        // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPStages; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&acc_full[i], 1);
      tc::mbar_init(&acc_empty[i], 4);   // the four epilogue warps
    }
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kPTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && my_tiles > 0) {
      tc::tma_prefetch(&tm_x);
      tc::tma_prefetch(&tm_w);
      const int total = my_tiles * nk;
      int issued = 0;
      for (int gi = 0; gi < total; ++gi) {
        const int tile = (int)blockIdx.x + (gi / nk) * (int)gridDim.x, kc = gi % nk;
        const int nt = tile % n_nt, mt = tile / n_nt;
        const int stage = gi % kPStages;
        const uint32_t round = uint32_t(gi / kPStages);
        if (!tc::mbar_wait_bounded(&empty[stage], (round & 1) ^ 1, abort_flag, a.wait_ns)) break;
        uint8_t* st = smem + stage * kPStageBytes;
        tc::mbar_arrive_expect_tx(&full[stage], kPAStage + b_bytes);
        tc::tma_load_2d(st, &tm_x, &full[stage], kc * kPChunk, mt * kPTile);
        tc::tma_load_2d(st + kPAStage, &tm_w, &full[stage], kc * kPChunk, nt * a.rank);
        ++issued;
      }
      if (issued < total) {
        // drain the copies still in flight before the CTA may exit
        volatile int quiet = 0;
        for (int gi = (issued > kPStages ? issued - kPStages : 0); gi < issued; ++gi)
          tc::mbar_wait_bounded(&full[gi % kPStages], uint32_t(gi / kPStages) & 1, &quiet, a.wait_ns / 10);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && my_tiles > 0) {
      const uint32_t idesc = tc::idesc_f16(kPTile, a.rank, P.bf16 != 0);
      const uint32_t base = tc::smem_addr(smem);
      bool ok = true;
      int gi = 0;
      uint64_t* last_bar = nullptr;   // the barrier of the last commit issued, and its phase parity
      uint32_t last_par = 0;
      for (int it = 0; it < my_tiles && ok; ++it) {
        const int buf = it & 1;
        if (!tc::mbar_wait_bounded(&acc_empty[buf], ((it >> 1) & 1) ^ 1, abort_flag, a.wait_ns)) break;
        tc::tc_fence_after();
        const uint32_t d = tmem_base + buf * kPAccCols;
        for (int kc = 0; kc < nk; ++kc, ++gi) {
          const int stage = gi % kPStages;
          if (!tc::mbar_wait_bounded(&full[stage], uint32_t(gi / kPStages) & 1, abort_flag, a.wait_ns)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t sa = base + stage * kPStageBytes;
#pragma unroll
          for (int k = 0; k < kPChunk / 16; ++k)
            tc::umma_f16(d, tc::sdesc_k_sw128(sa + k * 32), tc::sdesc_k_sw128(sa + kPAStage + k * 32), idesc,
                         (kc | k) != 0);
          tc::umma_commit(&empty[stage]);
          last_bar = &empty[stage];
          last_par = uint32_t(gi / kPStages) & 1;
        }
        if (!ok) break;
        tc::umma_commit(&acc_full[buf]);
        last_bar = &acc_full[buf];
        last_par = uint32_t(it >> 1) & 1;
      }
      // every MMA this thread issued has completed once its last commit lands
      if (last_bar) {
        volatile int quiet = 0;
        tc::mbar_wait_bounded(last_bar, last_par, &quiet, a.wait_ns);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    for (int it = 0; it < my_tiles; ++it) {
      const int buf = it & 1;
      const int tile = (int)blockIdx.x + it * (int)gridDim.x;
      const int nt = tile % n_nt, mt = tile / n_nt;
      const int side = nt / a.n_g, g = nt % a.n_g;
      const int64_t m = (int64_t)mt * kPTile + row;
      const bool got = tc::mbar_wait_bounded(&acc_full[buf], (it >> 1) & 1, abort_flag, a.wait_ns);
      if (!__all_sync(0xffffffffu, got)) break;   // a wait gave up: stop (the error is recorded below)
      tc::tc_fence_after();
      bool store = m < a.M;
      int64_t crow = 0;
      if (store) {
        const int b = int(m / a.n_new), t = int(m % a.n_new);
        const int64_t slot = (int64_t)a.dst_slot[b] + t;
        if (slot < 0 || slot >= a.capacity) {
          record_error(a.err, kCodeDevice, kErrSlot, int(slot), b);
          store = false;
        } else {
          crow = ((int64_t)b * a.capacity + slot) * a.n_g + g;
        }
      }
      write_row(a, tmem_base + (uint32_t(quad * 32) << 16) + buf * kPAccCols, side, crow, store);
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[buf]);
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (threadIdx.x == 0 && *abort_flag) record_error(a.err, kCodeTimeout, kErrWait, blockIdx.x, 0);
  if (warp == 1) tc::tmem_dealloc(tmem_base, kPTmemCols);
}

// W[side][g][m][e] = A_side[g][e][m] in the operand dtype: a 32 x 32 tiled transpose per (side, g)
template <typename IT, typename OT>
__global__ void prepare_down_proj_kernel(const IT* __restrict__ ak, const IT* __restrict__ av, OT* __restrict__ w,
                                         int n_g, int rank, int64_t d) {
  __shared__ float tile[32][33];
  const int sg = blockIdx.z, side = sg / n_g, g = sg % n_g;
  const IT* src = (side == 0 ? ak : av) + (int64_t)g * d * rank;   // [d][rank]
  OT* dst = w + (int64_t)sg * rank * d;                           // [rank][d]
  const int64_t e0 = (int64_t)blockIdx.x * 32;
  const int m0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;           // 32 x 8 threads
  for (int i = ty; i < 32; i += 8) {
    const int64_t e = e0 + i;
    const int m = m0 + tx;
    tile[i][tx] = (e < d && m < rank) ? to_f32(src[e * rank + m]) : 0.f;
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int m = m0 + i;
    const int64_t e = e0 + tx;
    if (m < rank && e < d) dst[(int64_t)m * d + e] = from_f32<OT>(tile[tx][i]);
  }
}

template <typename IT>
cudaError_t launch_prepare_typed(const void* ak, const void* av, int n_g, int rank, int64_t d, int w_dtype, void* w,
                                 cudaStream_t st) {
  dim3 grid((unsigned)((d + 31) / 32), (unsigned)((rank + 31) / 32), (unsigned)(2 * n_g));
  const IT* k = static_cast<const IT*>(ak);
  const IT* v = static_cast<const IT*>(av);
  if (w_dtype == kBF16)
    prepare_down_proj_kernel<IT, __nv_bfloat16><<<grid, 256, 0, st>>>(k, v, static_cast<__nv_bfloat16*>(w), n_g,
                                                                      rank, d);
  else
    prepare_down_proj_kernel<IT, __half><<<grid, 256, 0, st>>>(k, v, static_cast<__half*>(w), n_g, rank, d);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prepare_down_proj(const void* a_k, const void* a_v, int a_dtype, int n_g, int rank, int64_t d,
                                     int w_dtype, void* w, cudaStream_t st) {
  if (a_dtype == kF32) return launch_prepare_typed<float>(a_k, a_v, n_g, rank, d, w_dtype, w, st);
  if (a_dtype == kBF16) return launch_prepare_typed<__nv_bfloat16>(a_k, a_v, n_g, rank, d, w_dtype, w, st);
  return launch_prepare_typed<__half>(a_k, a_v, n_g, rank, d, w_dtype, w, st);
}

cudaError_t launch_project_latents(const void* x, const void* w, int bf16, const ProjectArgs& a, cudaStream_t st) {
  if (!tma_available()) return cudaErrorNotSupported;
  if (a.M == 0) return cudaSuccess;
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap tm_x, tm_w;
  {
    // x as [M][d]: boxes of 64 columns x 128 rows (rows past M read as zero)
    const cuuint64_t dims[2] = {(cuuint64_t)a.d, (cuuint64_t)a.M};
    const cuuint64_t strides[1] = {(cuuint64_t)a.d * 2};
    const cuuint32_t box[2] = {kPChunk, kPTile};
    if (!tma_encode(&tm_x, dt, 2, x, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  }
  {
    // W as [2 n_g r][d]: boxes of 64 columns x r rows
    const cuuint64_t dims[2] = {(cuuint64_t)a.d, (cuuint64_t)2 * a.n_g * a.rank};
    const cuuint64_t strides[1] = {(cuuint64_t)a.d * 2};
    const cuuint32_t box[2] = {kPChunk, (cuuint32_t)a.rank};
    if (!tma_encode(&tm_w, dt, 2, w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  }
  PrefillParams P;
  P.a = a;
  P.bf16 = bf16;
  cudaError_t e = cudaFuncSetAttribute(project_latents_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t n_tiles = (a.M + kPTile - 1) / kPTile * (2 * a.n_g);
  const unsigned grid = (unsigned)(n_tiles < sms ? n_tiles : sms);   // persistent: one CTA per SM
  project_latents_kernel<<<grid, kPThreads, kPSmem, st>>>(tm_x, tm_w, P);
  return cudaGetLastError();
}

}  // namespace palu
